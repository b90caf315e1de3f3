"""Host-side checks of libdsa that need no GPU: the library builds and loads,
exports every entry point dsa.h declares, and rejects bad arguments before
launching anything."""
import ctypes

import pytest

import __graft_entry__


@pytest.fixture(scope="module")
def api():
    __graft_entry__.build()
    from deepseek_sparse_attention_fp8_gb300 import api as a

    return a


def test_exports_every_declared_symbol(api):
    names = api.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(api.lib, n), f"libdsa.so does not export {n}"
    assert "sm_103a" in api.dsa_version()


def _null():
    return ctypes.c_void_p(0)


def test_indexer_rejects_bad_arguments(api):
    lib = api.lib
    st = lib.dsa_indexer_logits(_null(), 8192, _null(), _null(), 8448, 10, _null(), 4, _null(), _null(), 2, 2, 64,
                                128, 64, 1, _null(), 256, _null(), _null())
    assert st == api.DSA_ERR_INVALID_ARG
    assert b"null" in lib.dsa_last_error()
    st = lib.dsa_indexer_logits(_null(), 8192, _null(), _null(), 8448, 10, _null(), 4, _null(), _null(), -1, 2, 64,
                                128, 64, 1, _null(), 256, _null(), _null())
    assert st == api.DSA_ERR_INVALID_ARG
    # nothing to do: succeeds without touching a device
    st = lib.dsa_indexer_logits(_null(), 8192, _null(), _null(), 8448, 10, _null(), 4, _null(), _null(), 0, 0, 64,
                                128, 64, 1, _null(), 256, _null(), _null())
    assert st == api.DSA_OK


def test_indexer_shape_limits(api):
    lib = api.lib
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    args = lambda Hi, Di, bs, stride: (fake, Hi * Di, fake, fake, stride, 10, fake, 4, fake, fake, 1, 1, Hi, Di, bs, 1,
                                       fake, 256, _null(), _null())
    assert lib.dsa_indexer_logits(*args(65, 128, 64, 8448)) == api.DSA_ERR_UNSUPPORTED
    assert lib.dsa_indexer_logits(*args(64, 96, 64, 8448)) == api.DSA_ERR_UNSUPPORTED
    assert lib.dsa_indexer_logits(*args(64, 128, 32, 8448)) == api.DSA_ERR_UNSUPPORTED
    assert lib.dsa_indexer_logits(*args(64, 128, 64, 8000)) == api.DSA_ERR_INVALID_ARG


def test_topk_rejects_bad_arguments(api):
    lib = api.lib
    assert lib.dsa_topk(_null(), 100, _null(), _null(), 1, 1, 10, _null(), _null(), 0, _null()) == api.DSA_ERR_INVALID_ARG
    assert lib.dsa_topk(_null(), 100, _null(), _null(), 1, -1, 10, _null(), _null(), 0, _null()) == api.DSA_ERR_INVALID_ARG
    assert lib.dsa_topk(_null(), 100, _null(), _null(), 1, 0, 10, _null(), _null(), 0, _null()) == api.DSA_OK


def test_workspace_sizes(api):
    # the CTAs of a row combine their histograms in distributed shared memory
    for T, ld in ((32, 8192), (8, 131072), (4096, 65536), (1, 1 << 20)):
        assert api.dsa_topk_workspace_size(T, ld, 2048) == 0
    assert api.sparse_mla_workspace_size(32, 128, 512, 1) == 0
    assert api.sparse_mla_workspace_size(8, 128, 512, 8) == 8 * 128 * 8 * (512 * 4 + 8)


def test_auto_splits_heuristic(api):
    s_decode = api.sparse_mla_auto_splits(32, 128, 512, 2048)
    s_long = api.sparse_mla_auto_splits(8, 128, 512, 2048)
    s_many = api.sparse_mla_auto_splits(4096, 128, 512, 2048)
    assert 1 <= s_decode <= 32 and 1 <= s_long <= 32
    assert s_long >= s_decode  # fewer tokens -> more splits to fill the GPU
    assert s_many == 1


def test_mla_rejects_bad_arguments(api):
    lib = api.lib
    fake = ctypes.c_void_p(1 << 20)
    base = [fake, fake, 64 * 576, 10, fake, 4, fake, fake, fake, 1, 1, 128]
    tail = [2048, 64, 0.04, 0, fake, _null(), _null(), 0, _null(), _null()]
    assert lib.sparse_mla_decode(*base, 100, 64, *tail) == api.DSA_ERR_UNSUPPORTED
    assert lib.sparse_mla_decode(*(base[:11] + [129]), 576, 512, *tail) == api.DSA_ERR_UNSUPPORTED
    bad_scale = list(tail)
    bad_scale[2] = -1.0
    assert lib.sparse_mla_decode(*base, 576, 512, *bad_scale) == api.DSA_ERR_INVALID_ARG
    bad_splits = list(tail)
    bad_splits[3] = 33
    st = lib.sparse_mla_decode(*base, 576, 512, *bad_splits)
    assert st in (api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED, api.DSA_ERR_CUDA)
    null_q = [_null()] + base[1:]
    assert lib.sparse_mla_prefill(*null_q, 576, 512, 2048, 64, 0.04, fake, _null(), _null(), _null()) == \
        api.DSA_ERR_INVALID_ARG


def test_k_quant_and_cache_rejects_bad_arguments(api):
    lib = api.lib
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first

    def call(T=4, Di=128, bs=64, stride=64 * 132, k_stride=128, k=fake):
        return lib.dsa_indexer_k_quant_and_cache(k, k_stride, T, Di, fake, stride, 10, fake, 4, fake, fake, 1, bs,
                                                 _null(), _null())

    assert call(Di=48) == api.DSA_ERR_UNSUPPORTED
    assert call(bs=32) == api.DSA_ERR_UNSUPPORTED
    assert call(stride=64 * 132 - 16) == api.DSA_ERR_INVALID_ARG
    assert call(k_stride=100) == api.DSA_ERR_INVALID_ARG
    assert call(k=_null()) == api.DSA_ERR_INVALID_ARG
    assert b"null" in lib.dsa_last_error()
    assert call(T=-1) == api.DSA_ERR_INVALID_ARG
    assert call(T=0) == api.DSA_OK  # nothing to do: no device touched


def test_header_is_plain_c_and_links(api, tmp_path):
    """include/dsa.h compiles as pedantic C99 and a C program linked against
    libdsa.so gets the documented host-side answers (no GPU touched)."""
    import os
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    libdir = os.path.dirname(api.lib._name)
    exe = str(tmp_path / "c_abi_check")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(root, "include"),
                        os.path.join(here, "c_abi_check.c"), "-L", libdir, "-ldsa", f"-Wl,-rpath,{libdir}", "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)
