// Host-side helpers shared by the entry points: status/error reporting,
// device capability checks and launch checks.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/dsa.h"

namespace dsa {

// Records a formatted reason for dsa_last_error() and returns `st`.
dsa_status_t fail(dsa_status_t st, const char* fmt, ...);

// DSA_OK when the current device is an sm_103 part; sets the error otherwise.
dsa_status_t check_device();

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Encodes a tiled TMA descriptor (cuTensorMapEncodeTiled reached through the
// runtime's driver entry point, so the library does not link libcuda).
// dims/box are innermost first; strides_bytes has rank-1 entries.
dsa_status_t make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Converts a pending launch error into DSA_ERR_CUDA.
dsa_status_t check_launch(const char* what);

// Per-device record of which kernels have had their shared-memory
// attributes set. The flags are atomics and the first setting on a device is
// made under the mutex, so concurrent first calls and several devices in one
// process are both safe.
constexpr int kMaxDeviceOrdinals = 64;
struct FuncAttrOnce {
  std::mutex mu;
  std::atomic<bool> done[kMaxDeviceOrdinals] = {};
};

// Raises the dynamic shared-memory limit of a kernel once per device.
template <typename K>
dsa_status_t allow_smem(K kernel, int bytes, FuncAttrOnce& once) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDeviceOrdinals) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  if (once.done[dev].load(std::memory_order_acquire)) return DSA_OK;
  std::lock_guard<std::mutex> lock(once.mu);
  if (once.done[dev].load(std::memory_order_relaxed)) return DSA_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "cudaFuncSetAttribute(%d bytes): %s", bytes, cudaGetErrorString(e));
  // every kernel of the library asks for the same (largest) shared-memory
  // carveout, so consecutive launches never wait for the SMs to be re-split
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "cudaFuncSetAttribute(carveout): %s", cudaGetErrorString(e));
  once.done[dev].store(true, std::memory_order_release);
  return DSA_OK;
}

// The arguments of an indexer-logits call (a0 + a1), shared by the entry
// points that compute logits.
struct IndexerCall {
  const void* q_idx;
  int64_t q_stride_t;
  const float* w;
  const uint8_t* k_cache;
  int64_t k_block_stride_bytes;
  int32_t num_blocks;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t B, T, Hi, Di, block_size, max_q_len;
  int32_t* dev_status;
};
// Host-side checks of an indexer call (DSA_OK or the error, recorded).
dsa_status_t indexer_validate(const IndexerCall& c, const char* name);
// Enqueues the logits of keys [key_begin, key_begin + ld) into logits [T, ld]
// (column j = key key_begin + j); requests are clipped to keys below key_cap.
dsa_status_t indexer_launch(const IndexerCall& c, float* logits, int64_t ld, int64_t key_begin, int64_t key_cap,
                            cudaStream_t stream);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

constexpr float kNegSentinel = -1e30f;  // finite score of an empty / masked slot

// bits OR-ed into the caller's device status word
__device__ __forceinline__ void report(int32_t* dev_status, uint32_t bit) {
  if (dev_status != nullptr) atomicOr(reinterpret_cast<unsigned int*>(dev_status), bit);
}

}  // namespace dsa
