// tq_verify_noalloc: tq_verify with its scratch (partials, log-sum-exps and
// merge counters) in file-scope device arrays of this library instead of
// caller buffers, so that a call allocates nothing.  The pages have no
// counterpart of this entry point; it is a convenience of the C ABI.
//
// Set-up, once per device on the first call: the arrays' device addresses are
// looked up (cudaGetSymbolAddress) and the counters are cleared (the merge
// leaves them zero after every call).  Every call then forwards to tq_verify
// with those addresses, after checking that the problem fits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tqkv.h"
#include "tq_common.cuh"

namespace {

// partials [n_spec B Hq S][128] then log-sum-exps [n_spec B Hq S]: 16 MiB
constexpr size_t kScratchFloats = size_t(4) << 20;
// merge counters [B][Hk][4]
constexpr size_t kCounterWords = size_t(1) << 14;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];
static __device__ __align__(256) uint32_t g_noalloc_counters[kCounterWords];

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  bool ready = false;
  float* scratch = nullptr;
  uint32_t* counters = nullptr;
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// the current device's scratch, set up on first use (not capturable: the
// first call on a device must come before any stream capture)
tq_status device_scratch(DeviceScratch* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch& d = g_dev[dev];
  if (!d.ready) {
    void* s = nullptr;
    void* c = nullptr;
    if (cudaGetSymbolAddress(&s, g_noalloc_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&c, g_noalloc_counters) != cudaSuccess ||
        cudaMemset(c, 0, sizeof(g_noalloc_counters)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return TQ_ERR_CUDA;
    }
    d.scratch = static_cast<float*>(s);
    d.counters = static_cast<uint32_t*>(c);
    d.ready = true;
  }
  *out = d;
  return TQ_OK;
}

}  // namespace

void tq::noalloc_mark_stale() {
  std::lock_guard<std::mutex> lock(g_mu);
  for (DeviceScratch& d : g_dev) d.ready = false;
}

extern "C" tq_status tq_verify_noalloc(const tq_cache_desc* cache, const void* q, const int32_t* block_table,
                                       int32_t max_blocks, const int32_t* seq_lens, int32_t n_spec, int32_t B,
                                       int32_t Hq, int32_t num_kv_splits, int32_t causal, float* out,
                                       void* stream) {
  if (!cache) return TQ_ERR_INVALID_ARG;
  // sizes tq_verify rejects are passed on for its own status; only a valid
  // problem too large for the scratch is refused here
  if (n_spec >= 1 && B >= 1 && Hq >= 1 && num_kv_splits >= 1 && cache->num_kv_heads >= 1) {
    const size_t rows = (size_t)n_spec * (size_t)B * (size_t)Hq * (size_t)num_kv_splits;
    const size_t counters = (size_t)B * (size_t)cache->num_kv_heads * 4;
    if (rows > kScratchFloats / 129 || counters > kCounterWords) return TQ_ERR_UNSUPPORTED;
  }
  DeviceScratch d;
  const tq_status s = device_scratch(&d);
  if (s != TQ_OK) return s;
  const size_t rows = n_spec > 0 && B > 0 && Hq > 0 && num_kv_splits > 0
                          ? (size_t)n_spec * (size_t)B * (size_t)Hq * (size_t)num_kv_splits
                          : 0;
  return tq_verify(cache, q, block_table, max_blocks, seq_lens, n_spec, B, Hq, num_kv_splits, causal, d.scratch,
                   d.scratch + rows * 128, d.counters, out, stream);
}
