// Plain C++ oracle of the DeepSeek-Sparse-Attention step.
//
// TEST INFRASTRUCTURE ONLY: the test suite and the CPU-baseline legs of the
// benchmark load this library (built by build() into oracle/_build); the
// product path never does, and this file shares no code with it.
//
// It computes the plain definitions, one query token per task, in double
// precision, with std::thread over the tokens:
//   a0  per-(token, head) e4m3 quantisation of the indexer query
//       (scale = fp32(amax / 448), codes = e4m3 round-to-nearest-even,
//       saturating, of fp32(x / scale); amax == 0 gives scale 1)
//   a1  logits[t, s] = sum_h w[t,h] * ReLU( sum_d dq[t,h,d] * dk[s,d] ) for
//       s < valid(t), -inf up to ld; dq and dk are the fp8-decoded values
//       (code * scale), the sum is taken in double and rounded to fp32
//   a2  top-k of each row: the min(K, valid) largest values, equal values in
//       increasing position, -1 padding (a full sort)
//   a3  out[t,h,:] = sum_i softmax_i(scale * q[t,h,:] . kv[i,:]) kv[i,:Dv]
//       over the selected rows, lse = log sum_i exp(.), in double; no
//       selected row gives out 0 and lse -inf
// Sources (web pages, by title and section): vLLM PR #38476 "[Feature]
// TRITON_MLA_SPARSE backend for SM8x/11x/12x DSA Sparse MLA Support",
// Changes 2 (fp8 MQA logits, the K scale on the fp32 dot), Changes 3 (sparse
// MLA over the top-k rows), review thread (index_topk selection,
// per_token_group_quant_fp8 for the indexer q); "vllm-dsa-mtp-sm80" README,
// "The skew fixes" item 0 (the 132-byte indexer page, blocks addressed by the
// block stride). Readings where the pages are silent: a token sits at
// position seq_len - q_len + i and sees keys 0..pos; inside an indexer block,
// block_size rows of Di code bytes come first, then block_size fp32 scales;
// top-k values compare as floats (-0.0 equals +0.0); a top-k index is a
// logical position inside the request, mapped through the block table; the
// value vector is the first Dv dims of a latent row.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

double e4m3_value(uint8_t c) {
  const int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// Nearest e4m3 code of a finite value (ties to the even code), saturating at
// +-448: a search over the 127 non-negative finite codes, which are ordered.
uint8_t e4m3_code(double x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  uint8_t best = 0;
  for (int c = 1; c <= 0x7E; ++c) {
    const double dc = std::fabs(e4m3_value(static_cast<uint8_t>(c)) - a);
    const double db = std::fabs(e4m3_value(best) - a);
    if (dc < db || (dc == db && (c & 1) == 0)) best = static_cast<uint8_t>(c);
  }
  return sign | best;
}

double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

template <typename F>
void parallel_for(int n, int threads, F fn) {
  if (threads <= 1 || n <= 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w)
    pool.emplace_back([=]() {
      for (int i = w; i < n; i += threads) fn(i);
    });
  for (auto& th : pool) th.join();
}

struct Positions {
  std::vector<int64_t> req, pos;
};

Positions token_positions(const int32_t* seq_lens, const int32_t* qsl, int B) {
  Positions p;
  const int T = qsl[B];
  p.req.assign(T, 0);
  p.pos.assign(T, 0);
  for (int b = 0; b < B; ++b) {
    const int q_len = qsl[b + 1] - qsl[b];
    for (int i = 0; i < q_len; ++i) {
      p.req[qsl[b] + i] = b;
      p.pos[qsl[b] + i] = static_cast<int64_t>(seq_lens[b]) - q_len + i;
    }
  }
  return p;
}

}  // namespace

extern "C" {

// a0: codes [T*Hi, Di] and scales [T*Hi] of q (bf16 bits [T*Hi, Di]).
void oracle_quant_q(const uint16_t* q, int rows, int Di, uint8_t* codes, float* scales) {
  for (int r = 0; r < rows; ++r) {
    float amax = 0.f;
    for (int d = 0; d < Di; ++d) amax = std::max(amax, static_cast<float>(std::fabs(bf16_value(q[r * Di + d]))));
    const float scale = amax > 0.f ? amax / 448.0f : 1.0f;
    scales[r] = scale;
    for (int d = 0; d < Di; ++d) {
      const float y = static_cast<float>(bf16_value(q[r * Di + d])) / scale;
      codes[r * Di + d] = e4m3_code(y);
    }
  }
}

// a0 + a1 for the listed query tokens (others untouched): logits [T, ld].
void oracle_indexer_logits(const uint16_t* q_idx, const float* w, const uint8_t* k_cache, int64_t k_block_stride,
                           const int32_t* block_table, int bt_stride, const int32_t* seq_lens, const int32_t* qsl,
                           int B, int Hi, int Di, int block_size, int64_t ld, const int32_t* rows, int n_rows,
                           float* logits, int threads) {
  const Positions tp = token_positions(seq_lens, qsl, B);
  parallel_for(n_rows, threads, [&](int ri) {
    const int t = rows[ri];
    const int b = static_cast<int>(tp.req[t]);
    const int64_t valid = tp.pos[t] + 1;
    std::vector<uint8_t> qc(static_cast<size_t>(Hi) * Di);
    std::vector<float> qs(Hi);
    oracle_quant_q(q_idx + static_cast<int64_t>(t) * Hi * Di, Hi, Di, qc.data(), qs.data());
    std::vector<double> dq(static_cast<size_t>(Hi) * Di);
    for (int i = 0; i < Hi * Di; ++i) dq[i] = e4m3_value(qc[i]) * static_cast<double>(qs[i / Di]);
    std::vector<double> dk(Di);
    float* out = logits + static_cast<int64_t>(t) * ld;
    for (int64_t s = 0; s < ld; ++s) {
      if (s >= valid) {
        out[s] = -std::numeric_limits<float>::infinity();
        continue;
      }
      const int64_t blk = block_table[static_cast<int64_t>(b) * bt_stride + s / block_size];
      const uint8_t* page = k_cache + blk * k_block_stride;
      const int off = static_cast<int>(s % block_size);
      float ks;
      std::memcpy(&ks, page + static_cast<int64_t>(block_size) * Di + off * 4, 4);
      for (int d = 0; d < Di; ++d) dk[d] = e4m3_value(page[off * Di + d]) * static_cast<double>(ks);
      double acc = 0.0;
      for (int h = 0; h < Hi; ++h) {
        double dot = 0.0;
        for (int d = 0; d < Di; ++d) dot += dq[h * Di + d] * dk[d];
        acc += static_cast<double>(w[static_cast<int64_t>(t) * Hi + h]) * std::max(dot, 0.0);
      }
      out[s] = static_cast<float>(acc);
    }
  });
}

// a2 for the listed rows: topk [T, K] (largest first, ties by position).
void oracle_topk(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* qsl, int B, int K,
                 const int32_t* rows, int n_rows, int32_t* topk, int threads) {
  const Positions tp = token_positions(seq_lens, qsl, B);
  parallel_for(n_rows, threads, [&](int ri) {
    const int t = rows[ri];
    const int64_t n = std::min<int64_t>(tp.pos[t] + 1, ld);
    const float* row = logits + static_cast<int64_t>(t) * ld;
    std::vector<int32_t> idx(n);
    for (int64_t i = 0; i < n; ++i) idx[i] = static_cast<int32_t>(i);
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t c) { return row[a] > row[c]; });
    for (int k = 0; k < K; ++k) topk[static_cast<int64_t>(t) * K + k] = k < n ? idx[k] : -1;
  });
}

// a3 for the listed rows: out [T, H, Dv] and lse [T, H] in double.
void oracle_sparse_mla(const uint16_t* q, const uint16_t* kv_cache, int64_t kv_block_stride, const int32_t* block_table,
                       int bt_stride, const int32_t* seq_lens, const int32_t* qsl, int B, int H, int Dk, int Dv,
                       const int32_t* topk, int K, double softmax_scale, int block_size, const int32_t* rows,
                       int n_rows, double* out, double* lse, int threads) {
  const Positions tp = token_positions(seq_lens, qsl, B);
  parallel_for(n_rows, threads, [&](int ri) {
    const int t = rows[ri];
    const int b = static_cast<int>(tp.req[t]);
    std::vector<int64_t> sel;
    for (int k = 0; k < K; ++k) {
      const int32_t i = topk[static_cast<int64_t>(t) * K + k];
      if (i == -1) continue;
      const int64_t blk = block_table[static_cast<int64_t>(b) * bt_stride + i / block_size];
      sel.push_back(blk * kv_block_stride + static_cast<int64_t>(i % block_size) * Dk);
    }
    for (int h = 0; h < H; ++h) {
      double* o = out + (static_cast<int64_t>(t) * H + h) * Dv;
      if (sel.empty()) {
        for (int v = 0; v < Dv; ++v) o[v] = 0.0;
        lse[static_cast<int64_t>(t) * H + h] = -std::numeric_limits<double>::infinity();
        continue;
      }
      const uint16_t* qh = q + (static_cast<int64_t>(t) * H + h) * Dk;
      std::vector<double> s(sel.size());
      double m = -std::numeric_limits<double>::infinity();
      for (size_t j = 0; j < sel.size(); ++j) {
        double dot = 0.0;
        for (int d = 0; d < Dk; ++d) dot += bf16_value(qh[d]) * bf16_value(kv_cache[sel[j] + d]);
        s[j] = softmax_scale * dot;
        m = std::max(m, s[j]);
      }
      double z = 0.0;
      for (size_t j = 0; j < sel.size(); ++j) {
        s[j] = std::exp(s[j] - m);
        z += s[j];
      }
      for (int v = 0; v < Dv; ++v) o[v] = 0.0;
      for (size_t j = 0; j < sel.size(); ++j)
        for (int v = 0; v < Dv; ++v) o[v] += (s[j] / z) * bf16_value(kv_cache[sel[j] + v]);
      lse[static_cast<int64_t>(t) * H + h] = m + std::log(z);
    }
  });
}

int oracle_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? static_cast<int>(n) : 1;
}

}  // extern "C"
