// store_ops.cuh -- per (token, kv-head) quantise-and-pack of one new K/V
// token into its page ("spec-decode-intel-arc", section "Context": keys are
// Walsh-Hadamard rotated and coded against a Lloyd-Max codebook, or stored as
// FP8; values are uniform-scalar quantised with a scale and a zero).  One warp
// per token-head, lane l owning coordinates 4l .. 4l+3.  Shared by the store
// kernel and the single-launch store + verify, so that both write the same
// bytes.  All fp32 arithmetic uses explicitly rounded intrinsics (__fadd_rn,
// __fmul_rn, __fdiv_rn, __fsqrt_rn), so no step is contracted into an FMA:
//   |k|^2  = lane partial (x0^2 + x1^2) + (x2^2 + x3^2), then xor-butterfly
//            rounds at lane offsets 16, 8, 4, 2, 1;
//   H k    = unnormalised Sylvester butterflies, stride 1, 2 in-lane, then
//            strides 4..64 across lanes (offset stride / 4), (a + b, a - b);
//   y      = (H k) / (|k| * sqrt(128)),  code = #{boundaries strictly below y}
//            (7, 15 or 3 boundaries: 3-, 4- or 2-bit codes);
//   nc     = fp16(|k| / sqrt(|c_hat|^2)) with |c_hat|^2 summed in the same order.
#pragma once

#include <cuda_fp8.h>

#include "tq_common.cuh"

namespace tq {
namespace store_ops {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float half_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float tree_sum(float a0, float a1, float a2, float a3) {
  float s = __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(kFull, s, off));
  return s;
}

// fp16 -> e4m3, round to nearest even, saturating; NaN -> 0x7F.
__device__ __forceinline__ uint32_t e4m3_of_half(uint16_t h) {
  __half2_raw pair;
  pair.x = h;
  pair.y = 0;
  uint32_t b = (uint32_t)(__nv_cvt_halfraw2_to_fp8x2(pair, __NV_SATFINITE, __NV_E4M3) & 0xFFu);
  uint32_t mag = h & 0x7FFFu;
  if (mag > 0x7C00u) b = 0x7Fu;                        // NaN
  else if (mag == 0x7C00u) b = (h & 0x8000u) ? 0xFEu : 0x7Eu;  // +-inf saturates
  return b;
}

__device__ __forceinline__ void store_key8(uint8_t* page, int off, int lane, const uint16_t h[4]) {
  uint32_t w = e4m3_of_half(h[0]) | (e4m3_of_half(h[1]) << 8) | (e4m3_of_half(h[2]) << 16) |
               (e4m3_of_half(h[3]) << 24);
  *reinterpret_cast<uint32_t*>(page + K8::kKey + off * kD + 4 * lane) = w;
}

// coded keys, BITS = 3, 4 or 2 per coordinate (2^BITS-level codebook, page
// layout L); the fp16 key factor is |k| / |c_hat| (norm correction, the _nc
// presets) when corrected, else |k| (k3v4); bit i of signs flips the lane's
// coordinate i before the rotation (randomised-sign Hadamard, k3v4_nc_rs)
template <class L, int BITS>
__device__ __forceinline__ void store_keyq(uint8_t* page, int off, int lane, const uint16_t h[4],
                                           const Codebook& cb, bool corrected = true, uint32_t signs = 0u) {
  constexpr int N = 1 << BITS;
  float x[4], t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[i] = half_bits_to_float(h[i]);
    t[i] = ((signs >> i) & 1u) ? -x[i] : x[i];
  }
  const float ss = tree_sum(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1]), __fmul_rn(x[2], x[2]),
                            __fmul_rn(x[3], x[3]));
  const float norm = __fsqrt_rn(ss);
  // stride 1 and 2 inside the lane
  {
    float a = t[0], b = t[1];
    t[0] = __fadd_rn(a, b);
    t[1] = __fsub_rn(a, b);
    a = t[2];
    b = t[3];
    t[2] = __fadd_rn(a, b);
    t[3] = __fsub_rn(a, b);
    a = t[0];
    b = t[2];
    t[0] = __fadd_rn(a, b);
    t[2] = __fsub_rn(a, b);
    a = t[1];
    b = t[3];
    t[1] = __fadd_rn(a, b);
    t[3] = __fsub_rn(a, b);
  }
  // strides 4 .. 64 across lanes: the lower index holds a, the upper holds b
#pragma unroll
  for (int o = 1; o <= 16; o <<= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __shfl_xor_sync(kFull, t[i], o);
      t[i] = upper ? __fsub_rn(p, t[i]) : __fadd_rn(t[i], p);
    }
  }
  float C[N], Bd[N - 1];
#pragma unroll
  for (int m = 0; m < N; ++m) C[m] = half_bits_to_float(cb.c[m]);
#pragma unroll
  for (int m = 0; m < N - 1; ++m) Bd[m] = __fmul_rn(__fadd_rn(C[m], C[m + 1]), 0.5f);
  const float denom = __fmul_rn(norm, __fsqrt_rn(128.0f));
  uint32_t code[4];
  float c2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float y = (norm == 0.0f) ? 0.0f : __fdiv_rn(t[i], denom);
    uint32_t idx = 0;
#pragma unroll
    for (int m = 0; m < N - 1; ++m) idx += (y > Bd[m]) ? 1u : 0u;
    code[i] = idx;
    float c = C[0];
#pragma unroll
    for (int m = 1; m < N; ++m) c = (idx == (uint32_t)m) ? C[m] : c;
    c2[i] = __fmul_rn(c, c);
  }
  const float cn2 = tree_sum(c2[0], c2[1], c2[2], c2[3]);
  // 4 BITS bits per lane at stream bit 4 BITS lane of the token's 16 BITS bytes
  const uint32_t bits = code[0] | (code[1] << BITS) | (code[2] << (2 * BITS)) | (code[3] << (3 * BITS));
  uint8_t* kcodes = page + L::kKey + off * (16 * BITS);
  if constexpr (BITS == 4) {
    *reinterpret_cast<uint16_t*>(kcodes + 2 * lane) = (uint16_t)bits;
  } else if constexpr (BITS == 2) {
    kcodes[lane] = (uint8_t)bits;
  } else {
    // 12 bits per lane: 48 bytes = 12 little-endian words, word w gathered by lane w
    const int w = lane;
    uint64_t word = 0;
    const int first = (32 * w) / 12;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int src = min(first + j, 31);
      const uint32_t val = __shfl_sync(kFull, bits, src);
      const int shift = 12 * src - 32 * w;  // position of src's bits inside this word
      if (first + j <= 31 && shift > -12 && shift < 32) {
        word |= shift >= 0 ? ((uint64_t)val << shift) : ((uint64_t)val >> (-shift));
      }
    }
    if (lane < 12) *reinterpret_cast<uint32_t*>(kcodes + 4 * w) = (uint32_t)(word & 0xFFFFFFFFull);
  }
  if (lane == 0) {
    const uint16_t nc = !corrected ? __half_as_ushort(__float2half_rn(norm))
                        : (norm == 0.0f) ? (uint16_t)0
                                         : __half_as_ushort(__float2half_rn(__fdiv_rn(norm, __fsqrt_rn(cn2))));
    *reinterpret_cast<uint16_t*>(page + L::kNc + 2 * off) = nc;
  }
}

// the value quantiser of one (token, kv-head): writes its fp16 scale and
// zero (lane 0) and returns the 4-bit codes of the lane's 4 coordinates
template <class L>
__device__ __forceinline__ void value4_codes(uint8_t* page, int off, int lane, const uint16_t h[4], uint32_t c[4]) {
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = half_bits_to_float(h[i]);
  float lo = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
  float hi = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
  for (int off2 = 16; off2 >= 1; off2 >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(kFull, lo, off2));
    hi = fmaxf(hi, __shfl_xor_sync(kFull, hi, off2));
  }
  const __half zh = __float2half_rn(__fadd_rn(lo, 0.0f));  // -0 -> +0
  uint16_t sh = 0;
  if (hi != lo) {
    const float r = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    sh = __half_as_ushort(__float2half_rn(r));
    if (half_bits_to_float(sh) < r) sh = (uint16_t)(sh + 1);  // round the scale up
  }
  const float zf = __half2float(zh), sf = half_bits_to_float(sh);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float qv = 0.0f;
    if (sh != 0) qv = rintf(__fdiv_rn(__fsub_rn(v[i], zf), sf));
    qv = fminf(fmaxf(qv, 0.0f), 15.0f);
    c[i] = (uint32_t)qv;
  }
  if (lane == 0) {
    *reinterpret_cast<uint16_t*>(page + L::kScale + 2 * off) = sh;
    *reinterpret_cast<uint16_t*>(page + L::kZero + 2 * off) = __half_as_ushort(zh);
  }
}

// Value codes are stored coordinate-major: the 32-bit word vword(lane, i, off)
// of the value block holds coordinate 4 lane + i of tokens 8 (off / 8) ..
// 8 (off / 8) + 7, token off in bits vnib(off) .. vnib(off) + 3.
__device__ __forceinline__ int vword(int lane, int i, int off) { return 2 * (4 * lane + i) + (off >> 3); }
__device__ __forceinline__ int vnib(int off) { return 4 * (off & 7); }

template <class L>
__device__ __forceinline__ void store_value4(uint8_t* page, int off, int lane, const uint16_t h[4]) {
  uint32_t c[4];
  value4_codes<L>(page, off, lane, h, c);
  // tokens of one page share words, so each nibble is replaced atomically
  uint32_t* vw = reinterpret_cast<uint32_t*>(page + L::kVal);
  const int nib = vnib(off);
  const uint32_t keep = ~(0xFu << nib);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t* w = vw + vword(lane, i, off);
    atomicAnd(w, keep);
    atomicOr(w, c[i] << nib);
  }
}

// one (token, kv-head): 128 fp16 key and value coordinates (4 per lane, bits
// in kh / vh) into offset off of its page
// the 4 sign bits of lane's coordinates 4 lane .. 4 lane + 3
__device__ __forceinline__ uint32_t lane_signs(const uint32_t signs[4], int lane) {
  return (signs[lane >> 3] >> (4 * (lane & 7))) & 0xFu;
}

// the key of one (token, kv-head) for a kernel preset (0: FP8, else coded)
template <int PRESET>
__device__ __forceinline__ void store_key(uint8_t* page, int off, int lane, const uint16_t kh[4], const Codebook& cb,
                                          bool corrected, uint32_t signs) {
  if constexpr (PRESET == 0)
    store_key8(page, off, lane, kh);
  else
    store_keyq<Layout<PRESET>, key_bits<PRESET>()>(page, off, lane, kh, cb, corrected, signs);
}

template <int PRESET>
__device__ __forceinline__ void store_token(uint8_t* page, int off, int lane, const uint16_t kh[4],
                                            const uint16_t vh[4], const Codebook& cb, bool plain_norm = PRESET == 2,
                                            uint32_t signs = 0u) {
  using L = Layout<PRESET>;
  store_key<PRESET>(page, off, lane, kh, cb, !plain_norm, signs);
  store_value4<L>(page, off, lane, vh);
}

}  // namespace store_ops
}  // namespace tq
