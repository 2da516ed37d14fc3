// store.cu -- the fused store kernel of libtqkv: quantise and bit-pack new
// K/V tokens into the paged cache ("spec-decode-intel-arc", section
// "Context": the fused store is one of the three hot kernels).  One warp per
// (token, kv-head); the arithmetic is store_ops.cuh's.
#include "store_ops.cuh"

namespace tq {
namespace {

template <int PRESET>
__global__ void __launch_bounds__(128) store_kernel(StoreArgs a) {
  pdl_wait();
  pdl_trigger();
  using L = typename std::conditional<PRESET == 0, K8, K3>::type;
  const int lane = threadIdx.x & 31;
  const long unit = (long)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (unit >= (long)a.T * a.Hk) return;
  const long t = unit / a.Hk;
  const int h = (int)(unit % a.Hk);
  int32_t slot;
  if (a.slots) {
    slot = a.slots[t];
  } else {  // draft n of sequence b at position L_b - n_spec + n
    const int b = (int)(t / a.n_spec), n = (int)(t % a.n_spec);
    const int L = max(0, min(a.seq_lens[b], a.max_blocks * kBlock));
    const int pos = L - a.n_spec + n;
    const int id = pos >= 0 ? a.block_table[(long)b * a.max_blocks + pos / kBlock] : -1;
    slot = (id >= 0 && id < a.num_blocks) ? id * kBlock + pos % kBlock : -1;
  }
  if (slot < 0 || slot >= a.num_blocks * kBlock) return;  // skipped token (warp-uniform)
  const int blk = slot / kBlock, off = slot % kBlock;
  uint8_t* page = a.cache + ((long)blk * a.Hk + h) * L::kPage;
  const long base = (t * a.Hk + h) * kD + 4 * lane;
  const uint2 kr = *reinterpret_cast<const uint2*>(a.k + base);
  const uint2 vr = *reinterpret_cast<const uint2*>(a.v + base);
  const uint16_t kh[4] = {(uint16_t)(kr.x & 0xFFFF), (uint16_t)(kr.x >> 16), (uint16_t)(kr.y & 0xFFFF),
                          (uint16_t)(kr.y >> 16)};
  const uint16_t vh[4] = {(uint16_t)(vr.x & 0xFFFF), (uint16_t)(vr.x >> 16), (uint16_t)(vr.y & 0xFFFF),
                          (uint16_t)(vr.y >> 16)};
  store_ops::store_token<PRESET>(page, off, lane, kh, vh, a.cb);
}

}  // namespace

cudaError_t launch_store(int preset, const StoreArgs& a, cudaStream_t st) {
  const long units = (long)a.T * a.Hk;
  if (units == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((units + 3) / 4);
  if (preset == 0) return launch_pdl(store_kernel<0>, dim3(grid), dim3(128), 0, st, a);
  if (preset == 1) return launch_pdl(store_kernel<1>, dim3(grid), dim3(128), 0, st, a);
  return launch_pdl(store_kernel<2>, dim3(grid), dim3(128), 0, st, a);
}

}  // namespace tq
