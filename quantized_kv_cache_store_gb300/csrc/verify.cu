// verify.cu -- spec-verify attention over the quantised paged cache:
// stage 1 (split-KV partial attention) and stage 2 (log-sum-exp merge).
//
// Method ("spec-decode-intel-arc", sections "Part 3: The fused Triton
// kernel" and "Part 4: The causal correction"; "sycl-three-attempts-arc-b70",
// section "Part 3: joint_matrix + split-KV"): every draft query of a sequence
// is processed in one launch, one K dequant per cache tile is shared by all of
// them, scores are masked so draft n sees cached_len + n + 1 tokens, an online
// softmax keeps (m, l, acc) per query, the sequence is cut into NUM_KV_SPLITS
// ranges whose partials a second kernel merges by log-sum-exp.
//
// Stage 1 design (sm_103a): one CTA per (split, kv-head, sequence) holds ALL
// n_spec x (Hq / Hk) query rows of that kv-head, so each cache byte is read
// from HBM once.  Eight warps: RW row-warps (16 rows each) x TW token-groups.
// 16-token pages stream through a cp.async ring in shared memory; each warp
// dequantises its page straight from the ring into mma.sync fragments:
//   k8v4   : e4m3 -> f16 is exact (cvt f16x2.e4m3x2),
//   k3v4_nc: 3-bit codes -> fp16 centroids through a 64-entry pair table; the
//            per-token norm correction scales the score column after the MMA,
//            and the query is rotated once (q_rot = H q / sqrt(D), the
//            rotation's inverse moved to the query side);
//   values : 4-bit codes enter the MMA as exact small integers; the per-token
//            scale is folded into the probabilities (p * scale) and the zero
//            term sum_t p_t * zero_t is kept per row and added at the end.
// Token-groups merge their softmax states through shared memory at the end.
#include <math_constants.h>

#include <atomic>

#include <cuda_fp8.h>

#include "tq_common.cuh"

namespace tq {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// two e4m3 bytes (low 16 bits of w) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t w) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
  return (uint32_t)r.x | ((uint32_t)r.y << 16);
}

// one byte of value codes (two consecutive tokens of one coordinate: low
// nibble = even token) -> f16x2 of the two codes as exact integers 0..15
__device__ __forceinline__ uint32_t codepair_to_half2(uint32_t w, int byte) {
  const uint32_t b = (w >> (8 * byte)) & 0xFFu;
  const uint32_t magic = (b & 0xFu) | ((b & 0xF0u) << 12) | 0x64006400u;  // 1024 + n per half
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&magic),
                            __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int PAGE, int TW>
struct Ring {
  static constexpr int kStageBytes = TW * PAGE;
  static constexpr int kStages = (49152 / kStageBytes) < 4 ? 4 : (49152 / kStageBytes);
  static constexpr int kBytes = kStages * kStageBytes;
};

// Shared memory: ring | q (RW*16 x 128 fp16) | pair table (64 x u32)
template <int PRESET, int RW, int TW>
struct Smem {
  using L = Layout<PRESET>;
  using R = Ring<L::kPage, TW>;
  static constexpr int kMergeBytes = (TW - 1) * RW * (16 * kD + 48) * 4;
  static constexpr int kRingBytes = R::kBytes > kMergeBytes ? R::kBytes : kMergeBytes;
  static constexpr int kQOff = kRingBytes;
  static constexpr int kPairOff = kQOff + RW * 16 * kD * 2;
  static constexpr int kTotal = kPairOff + 64 * 4;
};

template <int PRESET, int RW, int TW>
__global__ void __launch_bounds__(RW* TW * 32, 1) verify_stage1_kernel(VerifyArgs a) {
  pdl_wait();
  pdl_trigger();
  using L = Layout<PRESET>;
  using RG = Ring<L::kPage, TW>;
  using SM = Smem<PRESET, RW, TW>;
  constexpr int NT = RW * TW * 32;
  constexpr int kChunks = L::kPage / 16;
  constexpr int kStages = RG::kStages;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  __half* qs = reinterpret_cast<__half*>(smem + SM::kQOff);
  uint32_t* pairs = reinterpret_cast<uint32_t*>(smem + SM::kPairOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rw = warp % RW, tg = warp / RW;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

  // ---- this split's token range
  int L_b = a.seq_lens[b];
  L_b = max(0, min(L_b, a.max_blocks * kBlock));
  const int per = (L_b + a.S - 1) / a.S;
  const int chunk = kBlock * ((per + kBlock - 1) / kBlock);
  const int t_lo = split * chunk;
  const int t_hi = min(t_lo + chunk, L_b);
  const int page_lo = t_lo / kBlock;
  const int npages = t_hi > t_lo ? (t_hi - t_lo + kBlock - 1) / kBlock : 0;
  const int niter = (npages + TW - 1) / TW;
  const int32_t* bt = a.block_table + (long)b * a.max_blocks;
  const uint8_t* cache_h = a.cache + (long)kvh * L::kPage;
  const long blk_stride = (long)a.Hk * L::kPage;

  auto issue = [&](int it) {
    if (it < niter) {
      uint8_t* dst = ring + (it % kStages) * RG::kStageBytes;
      for (int i = tid; i < TW * kChunks; i += NT) {
        const int p = it * TW + i / kChunks;
        if (p < npages) {
          const int blk = bt[page_lo + p];
          if (blk >= 0 && blk < a.num_blocks) {
            const int ch = i % kChunks;
            cp_async16(dst + (i / kChunks) * L::kPage + ch * 16, cache_h + blk * blk_stride + ch * 16);
          }
        }
      }
    }
    cp_async_commit();
  };

  // start streaming before the query prologue
#pragma unroll 1
  for (int it = 0; it < kStages - 1; ++it) issue(it);

  // ---- query prologue: rows r = n * group + j, rotated for k3v4_nc
  for (int rr = 0; rr < 16 / TW + (16 % TW ? 1 : 0); ++rr) {
    const int lr = tg + rr * TW;  // local row handled by this warp
    if (lr >= 16) break;
    const int r = rw * 16 + lr;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < a.R) {
      const int n = r / a.group, j = r % a.group;
      const __half* qp = a.q + (((long)n * a.B + b) * a.Hq + kvh * a.group + j) * kD + 4 * lane;
      const uint2 raw = *reinterpret_cast<const uint2*>(qp);
      const __half2 h0 = *reinterpret_cast<const __half2*>(&raw.x);
      const __half2 h1 = *reinterpret_cast<const __half2*>(&raw.y);
      x[0] = __low2float(h0);
      x[1] = __high2float(h0);
      x[2] = __low2float(h1);
      x[3] = __high2float(h1);
    }
    if (PRESET == 1) {
      // k3v4_nc_rs: q_rot = H diag(s) q / sqrt(128)
      const uint32_t sg = (a.signs[lane >> 3] >> (4 * (lane & 7))) & 0xFu;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if ((sg >> i) & 1u) x[i] = -x[i];
      float u = x[0], v = x[1];
      x[0] = u + v;
      x[1] = u - v;
      u = x[2];
      v = x[3];
      x[2] = u + v;
      x[3] = u - v;
      u = x[0];
      v = x[2];
      x[0] = u + v;
      x[2] = u - v;
      u = x[1];
      v = x[3];
      x[1] = u + v;
      x[3] = u - v;
#pragma unroll
      for (int o = 1; o <= 16; o <<= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float p = __shfl_xor_sync(kFull, x[i], o);
          x[i] = upper ? p - x[i] : x[i] + p;
        }
      }
      const float rs = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] *= rs;
    }
    uint2 out;
    out.x = pack_half2(x[0], x[1]);
    out.y = pack_half2(x[2], x[3]);
    *reinterpret_cast<uint2*>(qs + (rw * 16 + lr) * kD + 4 * lane) = out;
  }
  if (PRESET == 1 && tid < 64) {
    pairs[tid] = (uint32_t)a.cb.c[tid & 7] | ((uint32_t)a.cb.c[tid >> 3] << 16);
  }
  __syncthreads();

  // A fragments of this warp's 16 query rows: physical coordinate of logical
  // k-slot (kt, 2c + e) is 32c + 4kt + e, of (kt, 8 + 2c + e) is 32c + 4kt + 2 + e
  uint32_t qf[8][4];
  {
    const __half* ra = qs + (rw * 16 + g) * kD + 32 * c;
    const __half* rb = ra + 8 * kD;
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      const uint2 va = *reinterpret_cast<const uint2*>(ra + 4 * kt);
      const uint2 vb = *reinterpret_cast<const uint2*>(rb + 4 * kt);
      qf[kt][0] = va.x;
      qf[kt][1] = vb.x;
      qf[kt][2] = va.y;
      qf[kt][3] = vb.y;
    }
  }

  // rows of this thread and their visible limits inside the split
  const int rA = rw * 16 + g, rB = rA + 8;
  auto limit = [&](int r) {
    if (r >= a.R) return 0;
    const int n = r / a.group;
    const int vis = a.causal ? max(0, L_b - a.n_spec + n + 1) : L_b;
    return min(vis, t_hi);
  };
  const int limA = limit(rA), limB = limit(rB);

  float acc[16][4];
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
  float mA = -CUDART_INF_F, mB = -CUDART_INF_F, lA = 0.f, lB = 0.f, zA = 0.f, zB = 0.f;
  const float sl2 = kLog2e * 0.08838834764831845f;  // log2(e) / sqrt(128)

#pragma unroll 1
  for (int it = 0; it < niter; ++it) {
    issue(it + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const int p = it * TW + tg;
    if (p < npages) {
      const int blk = bt[page_lo + p];
      const bool valid = blk >= 0 && blk < a.num_blocks;
      const uint8_t* pg = ring + (it % kStages) * RG::kStageBytes + tg * L::kPage;
      const int pos0 = (page_lo + p) * kBlock;

      // ---- S = Q K^T for 16 tokens (two n-tiles of 8)
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        const int tok = nt * 8 + g;
        if constexpr (PRESET == 0) {
          const uint8_t* kr = pg + L::kKey + tok * kD + 32 * c;
          uint4 w[2];
          const int f = g & 1;  // alternate halves: conflict-free quarter-warps
          w[f] = *reinterpret_cast<const uint4*>(kr + 16 * f);
          w[f ^ 1] = *reinterpret_cast<const uint4*>(kr + 16 * (f ^ 1));
          const uint32_t ww[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
          for (int kt = 0; kt < 8; ++kt) {
            mma16816(s[nt], qf[kt], e4m3x2_to_half2(ww[kt]), e4m3x2_to_half2(ww[kt] >> 16));
          }
        } else {
          const uint32_t* kr = reinterpret_cast<const uint32_t*>(pg + L::kKey + tok * 48 + 12 * c);
          const uint32_t w0 = kr[0], w1 = kr[1], w2 = kr[2];
          const uint64_t lo64 = (uint64_t)w0 | ((uint64_t)w1 << 32);
          const uint64_t hi64 = (uint64_t)w1 | ((uint64_t)w2 << 32);
#pragma unroll
          for (int kt = 0; kt < 8; ++kt) {
            const uint32_t f12 = kt < 5 ? (uint32_t)(lo64 >> (12 * kt)) : (uint32_t)(hi64 >> (12 * kt - 32));
            const uint32_t b0 = pairs[f12 & 63];
            const uint32_t b1 = pairs[(f12 >> 6) & 63];
            mma16816(s[nt], qf[kt], b0, b1);
          }
        }
      }

      // ---- scale, mask, online softmax (log2 domain)
      // thread's tokens: nt*8 + 2c + e  (e = 0, 1)
      float colscale[2][2];
      if constexpr (PRESET == 1) {
        const uint32_t n0 = *reinterpret_cast<const uint32_t*>(pg + L::kNc + 2 * (2 * c));
        const uint32_t n1 = *reinterpret_cast<const uint32_t*>(pg + L::kNc + 2 * (8 + 2 * c));
        colscale[0][0] = __half2float(__ushort_as_half((uint16_t)(n0 & 0xFFFF))) * sl2;
        colscale[0][1] = __half2float(__ushort_as_half((uint16_t)(n0 >> 16))) * sl2;
        colscale[1][0] = __half2float(__ushort_as_half((uint16_t)(n1 & 0xFFFF))) * sl2;
        colscale[1][1] = __half2float(__ushort_as_half((uint16_t)(n1 >> 16))) * sl2;
      } else {
        colscale[0][0] = colscale[0][1] = colscale[1][0] = colscale[1][1] = sl2;
      }
      float mxA = -CUDART_INF_F, mxB = -CUDART_INF_F;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pos = pos0 + nt * 8 + 2 * c + e;
          const float va = (valid && pos < limA) ? s[nt][e] * colscale[nt][e] : -CUDART_INF_F;
          const float vb = (valid && pos < limB) ? s[nt][2 + e] * colscale[nt][e] : -CUDART_INF_F;
          s[nt][e] = va;
          s[nt][2 + e] = vb;
          mxA = fmaxf(mxA, va);
          mxB = fmaxf(mxB, vb);
        }
      mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 2));
      const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
      const float uA = nA == -CUDART_INF_F ? 0.f : nA;  // reference point (finite)
      const float uB = nB == -CUDART_INF_F ? 0.f : nB;
      if (__any_sync(kFull, nA > mA || nB > mB)) {
        const float aA = exp2f(mA - uA), aB = exp2f(mB - uB);
        lA *= aA;
        zA *= aA;
        lB *= aB;
        zB *= aB;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
          acc[dt][0] *= aA;
          acc[dt][1] *= aA;
          acc[dt][2] *= aB;
          acc[dt][3] *= aB;
        }
      }
      mA = nA;
      mB = nB;

      // value scale / zero of the thread's four tokens
      float vsc[2][2], vz[2][2];
      {
        const uint32_t s0 = *reinterpret_cast<const uint32_t*>(pg + L::kScale + 2 * (2 * c));
        const uint32_t s1 = *reinterpret_cast<const uint32_t*>(pg + L::kScale + 2 * (8 + 2 * c));
        const uint32_t z0 = *reinterpret_cast<const uint32_t*>(pg + L::kZero + 2 * (2 * c));
        const uint32_t z1 = *reinterpret_cast<const uint32_t*>(pg + L::kZero + 2 * (8 + 2 * c));
        vsc[0][0] = __half2float(__ushort_as_half((uint16_t)(s0 & 0xFFFF)));
        vsc[0][1] = __half2float(__ushort_as_half((uint16_t)(s0 >> 16)));
        vsc[1][0] = __half2float(__ushort_as_half((uint16_t)(s1 & 0xFFFF)));
        vsc[1][1] = __half2float(__ushort_as_half((uint16_t)(s1 >> 16)));
        vz[0][0] = __half2float(__ushort_as_half((uint16_t)(z0 & 0xFFFF)));
        vz[0][1] = __half2float(__ushort_as_half((uint16_t)(z0 >> 16)));
        vz[1][0] = __half2float(__ushort_as_half((uint16_t)(z1 & 0xFFFF)));
        vz[1][1] = __half2float(__ushort_as_half((uint16_t)(z1 >> 16)));
      }
      float pA[2][2], pB[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float ea = exp2f(s[nt][e] - uA), eb = exp2f(s[nt][2 + e] - uB);
          lA += ea;
          lB += eb;
          // a masked token contributes exactly 0 even if its unused slot
          // holds non-finite scale / zero bytes
          zA += ea > 0.f ? ea * vz[nt][e] : 0.f;
          zB += eb > 0.f ? eb * vz[nt][e] : 0.f;
          pA[nt][e] = ea > 0.f ? ea * vsc[nt][e] : 0.f;
          pB[nt][e] = eb > 0.f ? eb * vsc[nt][e] : 0.f;
        }
      uint32_t pf[4];
      pf[0] = pack_half2(pA[0][0], pA[0][1]);
      pf[1] = pack_half2(pB[0][0], pB[0][1]);
      pf[2] = pack_half2(pA[1][0], pA[1][1]);
      pf[3] = pack_half2(pB[1][0], pB[1][1]);

      // ---- O += P V: B fragment column n = g is coordinate d = 16g + dt; its
      // codes for tokens (2c, 2c+1) are byte c of the coordinate's 8-byte row,
      // for tokens (2c+8, 2c+9) byte 4 + c
      const uint2* vr = reinterpret_cast<const uint2*>(pg + L::kVal + 8 * 16 * g);
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        const uint2 row = vr[dt];
        mma16816(acc[dt], pf, codepair_to_half2(row.x, c), codepair_to_half2(row.y, c));
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- per-row totals over the quad
  lA += __shfl_xor_sync(kFull, lA, 1);
  lA += __shfl_xor_sync(kFull, lA, 2);
  lB += __shfl_xor_sync(kFull, lB, 1);
  lB += __shfl_xor_sync(kFull, lB, 2);
  zA += __shfl_xor_sync(kFull, zA, 1);
  zA += __shfl_xor_sync(kFull, zA, 2);
  zB += __shfl_xor_sync(kFull, zB, 1);
  zB += __shfl_xor_sync(kFull, zB, 2);

  // ---- merge token-groups through shared memory (ring is free now)
  if (TW > 1) {
    __syncthreads();
    float* mrg = reinterpret_cast<float*>(smem);
    constexpr int kSlot = 16 * kD + 48;
    if (tg > 0) {
      float* sl = mrg + ((tg - 1) * RW + rw) * kSlot;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        sl[g * kD + 32 * c + dt] = acc[dt][0];
        sl[g * kD + 32 * c + 16 + dt] = acc[dt][1];
        sl[(g + 8) * kD + 32 * c + dt] = acc[dt][2];
        sl[(g + 8) * kD + 32 * c + 16 + dt] = acc[dt][3];
      }
      if (c == 0) {
        float* st = sl + 16 * kD;
        st[g] = mA;
        st[g + 8] = mB;
        st[16 + g] = lA;
        st[16 + g + 8] = lB;
        st[32 + g] = zA;
        st[32 + g + 8] = zB;
      }
    }
    __syncthreads();
    if (tg == 0) {
#pragma unroll 1
      for (int o = 1; o < TW; ++o) {
        const float* sl = mrg + ((o - 1) * RW + rw) * kSlot;
        const float* st = sl + 16 * kD;
        const float m2A = st[g], m2B = st[g + 8];
        const float MA = fmaxf(mA, m2A), MB = fmaxf(mB, m2B);
        const float uA = MA == -CUDART_INF_F ? 0.f : MA, uB = MB == -CUDART_INF_F ? 0.f : MB;
        const float f1A = exp2f(mA - uA), f2A = exp2f(m2A - uA);
        const float f1B = exp2f(mB - uB), f2B = exp2f(m2B - uB);
        lA = lA * f1A + st[16 + g] * f2A;
        lB = lB * f1B + st[16 + g + 8] * f2B;
        zA = zA * f1A + st[32 + g] * f2A;
        zB = zB * f1B + st[32 + g + 8] * f2B;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
          acc[dt][0] = acc[dt][0] * f1A + sl[g * kD + 32 * c + dt] * f2A;
          acc[dt][1] = acc[dt][1] * f1A + sl[g * kD + 32 * c + 16 + dt] * f2A;
          acc[dt][2] = acc[dt][2] * f1B + sl[(g + 8) * kD + 32 * c + dt] * f2B;
          acc[dt][3] = acc[dt][3] * f1B + sl[(g + 8) * kD + 32 * c + 16 + dt] * f2B;
        }
        mA = MA;
        mB = MB;
      }
    }
  }
  if (tg != 0) return;

  // ---- write partials: o = (acc + zero term) / l, lse = ln(sum exp(score))
  auto write_row = [&](int r, float m, float l, float z, int half) {
    if (r >= a.R) return;
    const int n = r / a.group, j = r % a.group;
    const long row = (((long)n * a.B + b) * a.Hq + kvh * a.group + j) * a.S + split;
    float* o = a.part_o + row * kD + 32 * c;
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    float4 v[8];
    float* vv = reinterpret_cast<float*>(v);
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      vv[dt] = empty ? 0.f : (acc[dt][half] + z) * inv;
      vv[16 + dt] = empty ? 0.f : (acc[dt][half + 1] + z) * inv;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) reinterpret_cast<float4*>(o)[i] = v[i];
    if (c == 0) a.part_lse[row] = empty ? -CUDART_INF_F : (m + log2f(l)) * kLn2;
  };
  write_row(rA, mA, lA, zA, 0);
  write_row(rB, mB, lB, zB, 2);
}

// ---- stage 2: one warp per (n, b, h) row, lane owns 4 coordinates; lane s
// owns split s's weight exp(lse_s - M), broadcast while the partial rows of
// eight splits are loaded back to back
__global__ void __launch_bounds__(128) verify_stage2_kernel(MergeArgs a) {
  pdl_wait();
  pdl_trigger();
  const long row = (long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const float* lse = a.part_lse + row * a.S;
  float M = -CUDART_INF_F;
  for (int s = lane; s < a.S; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -CUDART_INF_F) {
    const float* po = a.part_o + row * a.S * kD + 4 * lane;
    float den = 0.f;
    for (int s0 = 0; s0 < a.S; s0 += 32) {
      const int s = s0 + lane;
      const float l = s < a.S ? lse[s] : -CUDART_INF_F;
      const float wl = l == -CUDART_INF_F ? 0.f : expf(l - M);
      den += wl;
      const int n = min(32, a.S - s0);
#pragma unroll 8
      for (int k = 0; k < n; ++k) {
        const float w = __shfl_sync(kFull, wl, k);
        const float4 v = *reinterpret_cast<const float4*>(po + (long)(s0 + k) * kD);
        if (w != 0.f) {  // an empty split contributes nothing
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
    const float inv = 1.f / den;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
  }
  *reinterpret_cast<float4*>(a.out + row * kD + 4 * lane) = acc;
}

template <int PRESET, int RW>
cudaError_t launch_s1(const VerifyArgs& a, cudaStream_t st) {
  constexpr int TW = 8 / RW;
  using SM = Smem<PRESET, RW, TW>;
  auto kern = verify_stage1_kernel<PRESET, RW, TW>;
  // the opt-in shared-memory size is a per-device function attribute
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kTotal);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  return launch_pdl(kern, dim3(a.S, a.Hk, a.B), dim3(RW * TW * 32), SM::kTotal, st, a);
}

template <int PRESET>
cudaError_t launch_s1_rows(const VerifyArgs& a, cudaStream_t st) {
  const int rw = (a.R + 15) / 16;
  if (rw <= 1) return launch_s1<PRESET, 1>(a, st);
  if (rw <= 2) return launch_s1<PRESET, 2>(a, st);
  if (rw <= 4) return launch_s1<PRESET, 4>(a, st);
  return launch_s1<PRESET, 8>(a, st);
}

}  // namespace

cudaError_t launch_verify_stage1(int preset, const VerifyArgs& a, cudaStream_t st) {
  if (verify_stage1_tc_supported(a)) return launch_verify_stage1_tc(preset, a, st);
  return preset == 0 ? launch_s1_rows<0>(a, st) : launch_s1_rows<1>(a, st);
}

cudaError_t launch_verify_stage2(const MergeArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((a.rows + 3) / 4);
  return launch_pdl(verify_stage2_kernel, dim3(grid), dim3(128), 0, st, a);
}

}  // namespace tq
