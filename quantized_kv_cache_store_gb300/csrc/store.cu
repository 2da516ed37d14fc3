// store.cu -- the fused store kernel of libtqkv: quantise and bit-pack new
// K/V tokens into the paged cache ("spec-decode-intel-arc", section
// "Context": the fused store is one of the three hot kernels).  One warp per
// (token, kv-head); the arithmetic is store_ops.cuh's.
#include "store_ops.cuh"

namespace tq {
namespace {

// slot of token t: slot_mapping[t], or for the drafts of a verify step the
// position min(seq_lens[b], max_blocks * 16) - n_spec + n through the block
// table (t = b * n_spec + n); -1 = skip
__device__ __forceinline__ int token_slot(const StoreArgs& a, long t) {
  if (a.slots) return a.slots[t];
  const int b = (int)(t / a.n_spec), n = (int)(t % a.n_spec);
  const int L = max(0, min(a.seq_lens[b], a.max_blocks * kBlock));
  const int pos = L - a.n_spec + n;
  const int id = pos >= 0 ? a.block_table[(long)b * a.max_blocks + pos / kBlock] : -1;
  return (id >= 0 && id < a.num_blocks) ? id * kBlock + pos % kBlock : -1;
}

// One CTA of 8 warps per (group of 8 consecutive tokens, kv-head), one warp
// per token.  When the group's slots are one aligned run of 8 (offsets
// 8g .. 8g + 7 of one page, as in a cache fill), the value-code words, which
// hold exactly those 8 tokens' nibbles, are merged in shared memory and
// written once with plain stores; otherwise each token's nibbles are replaced
// atomically in global memory (tokens of one page share words and may be
// written by other CTAs).
template <int PRESET>
__global__ void __launch_bounds__(256) store_kernel(StoreArgs a) {
  pdl_wait();
  pdl_trigger();
  using L = Layout<PRESET>;
  constexpr unsigned kFull = 0xffffffffu;
  __shared__ int slot8[8];
  __shared__ uint32_t words[128];  // the run's value words, coordinate-major
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long g = (long)blockIdx.x / a.Hk;
  const int h = (int)((long)blockIdx.x % a.Hk);
  const long t0 = g * 8;
  const int nt = (int)min(8L, (long)a.T - t0);
  if (threadIdx.x < 8) slot8[threadIdx.x] = (int)threadIdx.x < nt ? token_slot(a, t0 + threadIdx.x) : -1;
  if (threadIdx.x < 128) words[threadIdx.x] = 0u;
  __syncthreads();
  const int s0 = slot8[0];
  bool run8 = nt == 8 && s0 >= 0 && s0 < a.num_blocks * kBlock && (s0 & 7) == 0;
#pragma unroll
  for (int j = 1; j < 8; ++j) run8 = run8 && slot8[j] == s0 + j;
  const int slot = w < nt ? slot8[w] : -1;
  if (slot >= 0 && slot < a.num_blocks * kBlock) {  // warp-uniform
    const int blk = slot / kBlock, off = slot % kBlock;
    uint8_t* page = a.cache + ((long)blk * a.Hk + h) * L::kPage;
    const long base = ((t0 + w) * a.Hk + h) * kD + 4 * lane;
    const uint2 kr = *reinterpret_cast<const uint2*>(a.k + base);
    const uint2 vr = *reinterpret_cast<const uint2*>(a.v + base);
    const uint16_t kh[4] = {(uint16_t)(kr.x & 0xFFFF), (uint16_t)(kr.x >> 16), (uint16_t)(kr.y & 0xFFFF),
                            (uint16_t)(kr.y >> 16)};
    const uint16_t vh[4] = {(uint16_t)(vr.x & 0xFFFF), (uint16_t)(vr.x >> 16), (uint16_t)(vr.y & 0xFFFF),
                            (uint16_t)(vr.y >> 16)};
    if (run8) {
      store_ops::store_key<PRESET>(page, off, lane, kh, a.cb, a.plain_norm == 0, store_ops::lane_signs(a.signs, lane));
      uint32_t c[4];
      store_ops::value4_codes<L>(page, off, lane, vh, c);
#pragma unroll
      for (int i = 0; i < 4; ++i) atomicOr(&words[4 * lane + i], c[i] << store_ops::vnib(off));
    } else {
      store_ops::store_token<PRESET>(page, off, lane, kh, vh, a.cb, a.plain_norm != 0, store_ops::lane_signs(a.signs, lane));
    }
  }
  if (run8) {  // uniform across the CTA
    __syncthreads();
    if (w == 0) {
      uint32_t* vw = reinterpret_cast<uint32_t*>(a.cache + ((long)(s0 / kBlock) * a.Hk + h) * L::kPage + L::kVal);
#pragma unroll
      for (int i = 0; i < 4; ++i) vw[store_ops::vword(lane, i, s0 % kBlock)] = words[4 * lane + i];
    }
  }
}

}  // namespace

cudaError_t launch_store(int preset, const StoreArgs& a, cudaStream_t st) {
  const long units = ((long)a.T + 7) / 8 * a.Hk;  // (group of 8 tokens, kv-head): one CTA each
  if (units == 0) return cudaSuccess;
  const unsigned grid = (unsigned)units;
  // the k3 presets differ only in runtime flags (a.plain_norm, a.signs)
  switch (preset) {
    case 0: return launch_pdl(store_kernel<0>, dim3(grid), dim3(256), 0, st, a);
    case 4: return launch_pdl(store_kernel<4>, dim3(grid), dim3(256), 0, st, a);
    case 5: return launch_pdl(store_kernel<5>, dim3(grid), dim3(256), 0, st, a);
    default: return launch_pdl(store_kernel<1>, dim3(grid), dim3(256), 0, st, a);
  }
}

}  // namespace tq
