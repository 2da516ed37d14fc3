// tqkv_abi.cu -- the C ABI of libtqkv (declared in include/tqkv.h): argument
// validation, the codebook derivation and the kernel launches.  No entry point
// allocates, frees or synchronises; every check happens before any launch.
#include <cmath>
#include <cstdint>

#include "../../include/tqkv.h"
#include "tq_common.cuh"

namespace {

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// n-level Lloyd-Max quantiser of the standard normal (fp64, n = 4, 8, 16):
// alternate the nearest-neighbour condition (thresholds at midpoints of
// adjacent levels) and the centroid condition (each level is the mean of
// N(0,1) over its interval: (pdf(lo) - pdf(hi)) / (cdf(hi) - cdf(lo))) until
// no level moves by more than 1e-15.  The levels for N(0, 1/128) are these
// times 1/sqrt(128), rounded to fp16 ("spec-decode-intel-arc", section
// "Context": keys are coded against a precomputed Lloyd-Max codebook).
tq::Codebook derive_codebook(int n) {
  double y[16];
  for (int i = 0; i < n; ++i) y[i] = -2.0 + 4.0 * (i + 0.5) / n;  // uniform start
  auto pdf = [](double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) * 0.3989422804014327; };
  auto cdf = [](double x) {
    if (std::isinf(x)) return x > 0 ? 1.0 : 0.0;
    return 0.5 * std::erfc(-x * 0.7071067811865476);
  };
  auto sf = [](double x) {  // 1 - cdf, accurate in the upper tail
    if (std::isinf(x)) return x > 0 ? 0.0 : 1.0;
    return 0.5 * std::erfc(x * 0.7071067811865476);
  };
  for (int iter = 0; iter < 1000000; ++iter) {
    double t[17];
    t[0] = -INFINITY;
    t[n] = INFINITY;
    for (int i = 1; i < n; ++i) t[i] = 0.5 * (y[i - 1] + y[i]);
    double moved = 0.0;
    for (int i = 0; i < n; ++i) {
      const double lo = t[i], hi = t[i + 1];
      // probability mass of the cell, from whichever tail keeps precision
      const double mass = (lo >= 0.0) ? sf(lo) - sf(hi) : cdf(hi) - cdf(lo);
      const double ny = (pdf(lo) - pdf(hi)) / mass;
      moved = std::fmax(moved, std::fabs(ny - y[i]));
      y[i] = ny;
    }
    if (moved < 1e-15) break;
  }
  tq::Codebook cb = {};
  for (int i = 0; i < n; ++i) cb.c[i] = __half_as_ushort(__double2half(y[i] / std::sqrt(128.0)));
  return cb;
}

// levels of a preset's key codebook (0: FP8 keys or unknown)
int key_levels(int32_t preset) {
  switch (preset) {
    case TQ_PRESET_K3V4_NC:
    case TQ_PRESET_K3V4:
    case TQ_PRESET_K3V4_NC_RS: return 8;
    case TQ_PRESET_K4V4_NC: return 16;
    case TQ_PRESET_K2V4_NC: return 4;
    default: return 0;
  }
}

// the codebook of a coded-key preset (thread-safe one-time init per size)
const tq::Codebook& codebook(int32_t preset) {
  static const tq::Codebook c8 = derive_codebook(8), c16 = derive_codebook(16), c4 = derive_codebook(4);
  const int n = key_levels(preset);
  return n == 16 ? c16 : n == 4 ? c4 : c8;
}

// The sign vector of preset k3v4_nc_rs, as a mask (bit j set: s_j = -1):
// s_j = -1 where the top bit of output j of SplitMix64 (the output function
// published by Vigna) seeded with 0x54515F5349474E53 ("TQ_SIGNS") is set.
struct SignMask {
  uint32_t w[4];
};
SignMask rs_signs(int32_t preset) {
  SignMask m = {{0u, 0u, 0u, 0u}};
  if (preset != TQ_PRESET_K3V4_NC_RS) return m;
  for (int j = 0; j < 128; ++j) {
    uint64_t z = 0x54515F5349474E53ull + (uint64_t)(j + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    if (z >> 63) m.w[j >> 5] |= 1u << (j & 31);
  }
  return m;
}

bool is_k3(int32_t preset) {
  return preset == TQ_PRESET_K3V4_NC || preset == TQ_PRESET_K3V4 || preset == TQ_PRESET_K3V4_NC_RS;
}

size_t page_bytes(int32_t preset) {
  if (preset == TQ_PRESET_K8V4) return tq::K8::kPage;
  if (is_k3(preset)) return tq::K3::kPage;
  if (preset == TQ_PRESET_K4V4_NC) return tq::K4::kPage;
  if (preset == TQ_PRESET_K2V4_NC) return tq::K2::kPage;
  return 0;
}

tq_status check_desc(const tq_cache_desc* d) {
  if (!d || !d->cache) return TQ_ERR_INVALID_ARG;
  if (d->num_kv_heads < 1 || d->num_blocks < 0 || d->reserved != 0) return TQ_ERR_INVALID_ARG;
  if (page_bytes(d->preset) == 0) return TQ_ERR_UNSUPPORTED;
  if (d->head_dim != 128 || d->block_size != 16) return TQ_ERR_UNSUPPORTED;
  if (d->num_kv_heads > 65535) return TQ_ERR_UNSUPPORTED;
  if (!aligned(d->cache, 16)) return TQ_ERR_MISALIGNED;
  return TQ_OK;
}

tq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

// validation shared by tq_verify_stage1 and tq_verify; fills the kernel arguments
tq_status verify_args(const tq_cache_desc* cache, const void* q, const int32_t* block_table, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t n_spec, int32_t B, int32_t Hq, int32_t num_kv_splits,
                      int32_t causal, float* partial_o, float* partial_lse, tq::VerifyArgs* out_args) {
  tq_status s = check_desc(cache);
  if (s != TQ_OK) return s;
  if (!q || !block_table || !seq_lens || !partial_o || !partial_lse) return TQ_ERR_INVALID_ARG;
  if (n_spec < 1 || B < 0 || Hq < 1 || num_kv_splits < 1 || max_blocks < 1) return TQ_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return TQ_ERR_INVALID_ARG;
  if (Hq % cache->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
  const int group = Hq / cache->num_kv_heads;
  if (n_spec > 128 || n_spec * group > 1024) return TQ_ERR_UNSUPPORTED;
  const int rtiles = (n_spec * group + 63) / 64;
  if (num_kv_splits > 65535 || (long)B * rtiles > 65535 || max_blocks > (1 << 26)) return TQ_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(partial_o, 16) ||
      !aligned(partial_lse, 4))
    return TQ_ERR_MISALIGNED;
  tq::VerifyArgs& a = *out_args;
  a.cache = static_cast<const uint8_t*>(cache->cache);
  a.num_blocks = cache->num_blocks;
  a.Hk = cache->num_kv_heads;
  a.q = static_cast<const __half*>(q);
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.n_spec = n_spec;
  a.B = B;
  a.Hq = Hq;
  a.group = group;
  a.R = n_spec * group;
  a.rtiles = rtiles;
  a.S = num_kv_splits;
  a.causal = causal;
  a.part_o = partial_o;
  a.part_lse = partial_lse;
  a.out = nullptr;
  a.tickets = nullptr;
  a.dk = nullptr;
  a.dv = nullptr;
  a.cache_w = nullptr;
  a.plain_norm = cache->preset == TQ_PRESET_K3V4 ? 1 : 0;
  {
    const SignMask m = rs_signs(cache->preset);
    for (int i = 0; i < 4; ++i) a.signs[i] = m.w[i];
  }
  a.cb = codebook(cache->preset);
  return TQ_OK;
}

}  // namespace

extern "C" {

size_t tq_page_bytes(int32_t preset) { return page_bytes(preset); }

size_t tq_partials_bytes(int32_t n_spec, int32_t B, int32_t Hq, int32_t num_kv_splits) {
  if (n_spec < 1 || B < 1 || Hq < 1 || num_kv_splits < 1) return 0;
  return (size_t)n_spec * (size_t)B * (size_t)Hq * (size_t)num_kv_splits * (128 + 1) * sizeof(float);
}

int32_t tq_key_levels(int32_t preset) { return key_levels(preset); }

tq_status tq_codebook(int32_t preset, float* centroids_out) {
  if (!centroids_out) return TQ_ERR_INVALID_ARG;
  const int n = key_levels(preset);
  if (n == 0) return preset == TQ_PRESET_K8V4 ? TQ_ERR_UNSUPPORTED : TQ_ERR_INVALID_ARG;
  const tq::Codebook& cb = codebook(preset);
  for (int i = 0; i < n; ++i) centroids_out[i] = __half2float(__ushort_as_half(cb.c[i]));
  return TQ_OK;
}

const char* tq_status_string(int32_t status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument (null pointer, negative or inconsistent size)";
    case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case TQ_ERR_MISALIGNED: return "misaligned pointer";
    case TQ_ERR_CUDA: return "CUDA launch error";
    case TQ_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

tq_status tq_store(const tq_cache_desc* cache, const void* k, const void* v, const int32_t* slot_mapping,
                   int32_t T, void* stream) {
  tq_status s = check_desc(cache);
  if (s != TQ_OK) return s;
  if (T < 0) return TQ_ERR_INVALID_ARG;
  if (T == 0) return TQ_OK;
  if (!k || !v || !slot_mapping) return TQ_ERR_INVALID_ARG;
  if ((long)cache->num_blocks * 16 > INT32_MAX) return TQ_ERR_UNSUPPORTED;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 4)) return TQ_ERR_MISALIGNED;
  tq::StoreArgs a;
  a.cache = static_cast<uint8_t*>(cache->cache);
  a.num_blocks = cache->num_blocks;
  a.Hk = cache->num_kv_heads;
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.slots = slot_mapping;
  a.T = T;
  a.block_table = nullptr;
  a.max_blocks = 0;
  a.seq_lens = nullptr;
  a.n_spec = 0;
  a.plain_norm = cache->preset == TQ_PRESET_K3V4 ? 1 : 0;
  {
    const SignMask m = rs_signs(cache->preset);
    for (int i = 0; i < 4; ++i) a.signs[i] = m.w[i];
  }
  a.cb = codebook(cache->preset);
  return from_cuda(tq::launch_store(cache->preset, a, static_cast<cudaStream_t>(stream)));
}

tq_status tq_verify_stage1(const tq_cache_desc* cache, const void* q, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* seq_lens, int32_t n_spec, int32_t B,
                           int32_t Hq, int32_t num_kv_splits, int32_t causal, float* partial_o,
                           float* partial_lse, void* stream) {
  tq::VerifyArgs a;
  const tq_status s = verify_args(cache, q, block_table, max_blocks, seq_lens, n_spec, B, Hq, num_kv_splits,
                                  causal, partial_o, partial_lse, &a);
  if (s != TQ_OK || B == 0) return s;
  return from_cuda(tq::launch_verify_stage1(cache->preset, a, static_cast<cudaStream_t>(stream)));
}

tq_status tq_verify(const tq_cache_desc* cache, const void* q, const int32_t* block_table, int32_t max_blocks,
                    const int32_t* seq_lens, int32_t n_spec, int32_t B, int32_t Hq, int32_t num_kv_splits,
                    int32_t causal, float* partial_o, float* partial_lse, uint32_t* tickets, float* out,
                    void* stream) {
  tq::VerifyArgs a;
  tq_status s = verify_args(cache, q, block_table, max_blocks, seq_lens, n_spec, B, Hq, num_kv_splits, causal,
                            partial_o, partial_lse, &a);
  if (s != TQ_OK) return s;
  if (!out || !tickets) return TQ_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(tickets, 4)) return TQ_ERR_MISALIGNED;
  if (B == 0) return TQ_OK;
  a.out = out;
  a.tickets = tickets;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (tq::verify_fused_supported(cache->preset, a)) return from_cuda(tq::launch_verify_fused(cache->preset, a, st));
  s = from_cuda(tq::launch_verify_stage1(cache->preset, a, st));
  if (s != TQ_OK) return s;
  return tq_verify_stage2(partial_o, partial_lse, n_spec, B, Hq, 128, num_kv_splits, out, stream);
}



tq_status tq_store_verify(const tq_cache_desc* cache, const void* k_new, const void* v_new, const void* q,
                          const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, int32_t n_spec,
                          int32_t B, int32_t Hq, int32_t num_kv_splits, int32_t causal, float* partial_o,
                          float* partial_lse, uint32_t* tickets, float* out, void* stream) {
  tq::VerifyArgs a;
  tq_status s = verify_args(cache, q, block_table, max_blocks, seq_lens, n_spec, B, Hq, num_kv_splits, causal,
                            partial_o, partial_lse, &a);
  if (s != TQ_OK) return s;
  if (!out || !tickets || !k_new || !v_new) return TQ_ERR_INVALID_ARG;
  if ((long)cache->num_blocks * 16 > INT32_MAX) return TQ_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(tickets, 4) || !aligned(k_new, 16) || !aligned(v_new, 16))
    return TQ_ERR_MISALIGNED;
  if (B == 0) return TQ_OK;
  a.out = out;
  a.tickets = tickets;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (tq::verify_fused_supported(cache->preset, a)) {
    a.dk = static_cast<const __half*>(k_new);
    a.dv = static_cast<const __half*>(v_new);
    a.cache_w = static_cast<uint8_t*>(cache->cache);
    return from_cuda(tq::launch_verify_fused(cache->preset, a, st));
  }
  // otherwise the drafts go through the store kernel (slots from the block
  // table), then tq_verify
  tq::StoreArgs sa;
  sa.cache = static_cast<uint8_t*>(cache->cache);
  sa.num_blocks = cache->num_blocks;
  sa.Hk = cache->num_kv_heads;
  sa.k = static_cast<const __half*>(k_new);
  sa.v = static_cast<const __half*>(v_new);
  sa.slots = nullptr;
  sa.T = n_spec * B;
  sa.block_table = block_table;
  sa.max_blocks = max_blocks;
  sa.seq_lens = seq_lens;
  sa.n_spec = n_spec;
  sa.plain_norm = a.plain_norm;
  for (int i = 0; i < 4; ++i) sa.signs[i] = a.signs[i];
  sa.cb = codebook(cache->preset);
  s = from_cuda(tq::launch_store(cache->preset, sa, st));
  if (s != TQ_OK) return s;
  return tq_verify(cache, q, block_table, max_blocks, seq_lens, n_spec, B, Hq, num_kv_splits, causal, partial_o,
                   partial_lse, tickets, out, stream);
}

tq_status tq_verify_stage2(const float* partial_o, const float* partial_lse, int32_t n_spec, int32_t B,
                           int32_t Hq, int32_t head_dim, int32_t num_kv_splits, float* out, void* stream) {
  if (!partial_o || !partial_lse || !out) return TQ_ERR_INVALID_ARG;
  if (n_spec < 1 || B < 0 || Hq < 1 || num_kv_splits < 1) return TQ_ERR_INVALID_ARG;
  if (head_dim != 128) return TQ_ERR_UNSUPPORTED;
  if (!aligned(partial_o, 16) || !aligned(partial_lse, 4) || !aligned(out, 16)) return TQ_ERR_MISALIGNED;
  tq::MergeArgs a;
  a.part_o = partial_o;
  a.part_lse = partial_lse;
  a.out = out;
  a.rows = (long)n_spec * B * Hq;
  a.S = num_kv_splits;
  if ((a.rows + 3) / 4 > INT32_MAX) return TQ_ERR_UNSUPPORTED;
  return from_cuda(tq::launch_verify_stage2(a, static_cast<cudaStream_t>(stream)));
}

tq_status tq_device_status(void) {
  unsigned int word = 0;
  if (tq::read_device_error(&word, true) != cudaSuccess) return TQ_ERR_CUDA;
  if (word) tq::noalloc_mark_stale();
  return word ? TQ_ERR_TIMEOUT : TQ_OK;
}

}  // extern "C"
