// verify_tc.cu -- spec-verify stage 1 on the sm_103a tensor cores (tcgen05,
// tensor memory, TMA / bulk copies, mbarriers), for up to 64 query rows per
// kv-head.
//
// Method ("spec-decode-intel-arc", sections "Part 3: The fused Triton
// kernel" and "Part 4: The causal correction"; split-KV of
// "sycl-three-attempts-arc-b70", section "Part 3"): for one (split, kv-head,
// sequence) every draft x GQA query row attends to the split's visible cache
// tokens with an online softmax; one dequantisation of each cache tile serves
// all rows.
//
// Work is cut into chunks of 128 tokens (8 pages).  Both contractions are
// transposed so that the 128-row side of the MMA is tokens or coordinates:
//   S^T[token, row]  = K_hat[token, :] . Q[row, :]         (M = 128, N = rows)
//   O^T[d, row]     += V_codes^T[d, token] . P'[row, token] (M = 128, N = rows)
// with A operands in tensor memory (written by the worker threads with
// tcgen05.st) and B operands in shared memory (Q once per CTA; P' per chunk).
//   keys   : k8v4 e4m3 -> f16 exactly (the key block of a page arrives by TMA
//            with 128-byte swizzle, so the per-token row reads are free of
//            bank conflicts); k3v4_nc 3-bit code pairs -> fp16 centroid pairs
//            through a per-lane replicated table; the norm correction nc_t
//            scales token t's scores (its TMEM lane) after the MMA; the query
//            is rotated once, q_rot = H q / sqrt(D).
//   values : codes enter as exact fp16 subnormals (code * 2^-24, undone on
//            the output); P' = p * scale_t; the zero term sum_t p_t zero_t and
//            l = sum_t p_t are kept per thread in fp32, reduced at the end.
// Softmax: thread t owns token t (its S^T lane) and 16 query rows.  The
// running maximum is updated lazily: only when some score exceeds it by more
// than 8 (log2 units) is the exact chunk maximum computed across the 128
// tokens and O^T, l and the zero term rescaled; otherwise probabilities stay
// bounded by 2^8 and the stale maximum is used (any reference point gives the
// same softmax).
//
// Warp roles: warp 0 = producer (block ids + copies), warp 1 = MMA issuer,
// warp 2 = TMEM owner.  Worker warpgroup j (NMMA / 16 of them) dequantises its
// share of chunk c (A_K columns and A_V columns [64/W j, 64/W (j+1)); A_V is
// triple-buffered so that chunk c does not wait for O^T(c - 1)) and then
// runs the softmax of chunk c - 1 for query rows [16 j, 16 j + 16), so every
// scheduler keeps several warps busy.  Every wait on an mbarrier is bounded:
// on expiry the CTA sets an abort flag and the sticky device error word,
// drains its in-flight copies and MMAs, frees its tensor memory and writes
// NaN partials.
#include <math_constants.h>

#include <atomic>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include "tc_ptx.cuh"
#include "tq_common.cuh"

namespace tq {

__device__ unsigned int g_tq_device_error;  // sticky: nonzero after a bounded wait expired

namespace {

using namespace ptx;

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// a bounded wait gives up after kWaitTries tests of up to kSuspendNs each (~1 s)
constexpr uint32_t kWaitTries = 50000;
constexpr uint32_t kSuspendNs = 20000;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int PRESET, int NMMA>
struct Cfg {
  using L = Layout<PRESET>;
  static constexpr int kTok = 128;  // tokens per chunk
  static constexpr int kPages = 8;  // pages per chunk
  // k8v4 stage: the 8 key blocks [16][128] (TMA, 128B swizzle, 1024-aligned)
  // then the remaining 1088 bytes of each page; k3v4_nc stage: pages verbatim
  static constexpr int kKeyBlock = 16 * kD;
  static constexpr int kRestBytes = L::kPage - kKeyBlock;
  static constexpr int kRestOff = kPages * kKeyBlock;
  static constexpr int kStageBytes = align_up(kPages * L::kPage, 1024);
  static constexpr int kStages = PRESET == 0 ? 4 : 6;
  static constexpr int kW = NMMA / 16;   // worker warpgroups
  static constexpr int kNC = 16;         // query rows per worker thread
  static constexpr int kKC = 64 / kW;    // A-operand columns each worker warpgroup writes
  static constexpr int kThreads = 128 + 128 * kW;
  // per-thread register budgets after setmaxnreg (control / workers); their
  // sum must stay within what the launch granted (checked at launch)
  static constexpr int kRegCtl = 32;
  static constexpr int kRegW = kW == 4 ? 112 : (kW == 2 ? 200 : 232);
  static constexpr int kRegNeeded = 128 * kRegCtl + 128 * kW * kRegW;
  static constexpr int kLine = 2 * NMMA;  // bytes of one P' line (one token)
  static constexpr int kSwzBits = NMMA == 64 ? 3 : (NMMA == 32 ? 2 : 1);
  static constexpr uint32_t kSwzMode = NMMA == 64 ? 2u : (NMMA == 32 ? 4u : 6u);
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kRing = 0;
  static constexpr int kQ = align_up(kStages * kStageBytes, 1024);
  static constexpr int kQBytes = 2 * NMMA * 128;  // K-major, 128B swizzle, 2 x 64-coordinate blocks
  static constexpr int kP = kQ + align_up(kQBytes, 1024);
  static constexpr int kPBytes = kTok * kLine;  // one buffer
  static constexpr int kCol = kP + 2 * kPBytes;  // float4 [3][128]: column scale, v scale, v zero, row mask
  static constexpr int kRed = kCol + 3 * kTok * 16;  // float [kW][3][4][16], then float [kW][3][16]
  static constexpr int kPair = kRed + kW * 3 * 5 * kNC * 4;  // u32 [64][32] (k3v4_nc)
  static constexpr int kPValid = kPair + (PRESET == 1 ? 64 * 32 * 4 : 0);  // u8 [kStages][8]
  static constexpr int kBar = align_up(kPValid + kStages * 8, 8);
  // full[kStages] empty[kStages] akv[2] qk[2] sfree[2] pfull[2] pv[2]
  static constexpr int kNumBars = 2 * kStages + 10;
  static constexpr int kMisc = kBar + 8 * kNumBars;  // u32 tmem base, u32 abort
  static constexpr int kSmem = kMisc + 16 + 1024;    // + alignment slack
  // tensor memory columns
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTAK = 0;     // A_K[2]: 64 cols each (token lanes, coordinate pairs)
  static constexpr uint32_t kTAV = 128;   // A_V[3]: 64 cols each (coordinate lanes, token pairs)
  static constexpr uint32_t kTS = 320;    // S^T[2]: NMMA cols each
  static constexpr uint32_t kTO = 320 + 2 * NMMA;  // O^T: NMMA cols
  static_assert(kTO + NMMA <= kTmemCols, "tensor memory overflow");
  static_assert(kSmem <= 227 * 1024, "shared memory overflow");
};

struct Bars {
  uint32_t base;
  int stages;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (stages + s); }
  __device__ uint32_t akv(int b) const { return base + 8 * (2 * stages + b); }        // A operands + token params
  __device__ uint32_t qk(int b) const { return base + 8 * (2 * stages + 2 + b); }     // S^T = K Q^T done
  __device__ uint32_t sfree(int b) const { return base + 8 * (2 * stages + 4 + b); }  // S^T read by softmax
  __device__ uint32_t pfull(int b) const { return base + 8 * (2 * stages + 6 + b); }  // P' written
  __device__ uint32_t pv(int b) const { return base + 8 * (2 * stages + 8 + b); }     // O^T += V^T P'^T done
};

// Bounded wait; false when the CTA aborted or this wait expired (which aborts).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                         bool honour_abort = true) {
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
    if (honour_abort && *abort) return false;
    if (i >= kWaitTries) {
      *abort = 1u;
      atomicOr(&g_tq_device_error, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t w16) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w16 & 0xFFFFu), __NV_E4M3);
  return (uint32_t)r.x | ((uint32_t)r.y << 16);
}

// 2^x, hardware approximation (relative error ~2^-22), -inf -> 0
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Reduce NC values per lane across the 32 lanes of a warp; afterwards lane l
// holds the reduction of column (l % NC) in v[0].
template <int NC, bool MAX>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[NC], int lane) {
#pragma unroll
  for (int o = NC / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(kFull, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  if (NC < 32) {
#pragma unroll
    for (int o = 16; o >= NC; o >>= 1) {
      const float recv = __shfl_xor_sync(kFull, v[0], o);
      v[0] = MAX ? fmaxf(v[0], recv) : v[0] + recv;
    }
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 16) {
    tmem_st<16>(taddr, r);
  } else {
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
      uint32_t q[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) q[k] = r[32 * h + k];
      tmem_st<32>(taddr + 32 * h, q);
    }
  }
}

template <int PRESET, int NMMA>
__global__ void __launch_bounds__(Cfg<PRESET, NMMA>::kThreads, 1)
    verify_stage1_tc_kernel(VerifyArgs a, const __grid_constant__ CUtensorMap tmap_keys) {
  using C = Cfg<PRESET, NMMA>;
  using L = typename C::L;
  constexpr int kNC = C::kNC, kKC = C::kKC;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  uint8_t* pvalid = sm + C::kPValid;
  float4* colp = reinterpret_cast<float4*>(sm + C::kCol);
  float* red = reinterpret_cast<float*>(sm + C::kRed);
  uint32_t* pairs = reinterpret_cast<uint32_t*>(sm + C::kPair);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + C::kMisc + 4);
  const Bars bars{sbase + C::kBar, C::kStages};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  const int nchunks = (npages + C::kPages - 1) / C::kPages;
  const int32_t* bt = a.block_table + (long)b * a.max_blocks;

  // ---- set-up: barriers, tensor memory
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 4 * C::kW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.akv(i), 4 * C::kW);
      mbar_init(bars.qk(i), 1);
      mbar_init(bars.sfree(i), 4 * C::kW);
      mbar_init(bars.pfull(i), 4 * C::kW);
      mbar_init(bars.pv(i), 1);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();  // barriers initialised

  // Producer = warp 0 (all lanes wait together; lane 0 issues the copies).
  // Block ids are fetched 32 pages (4 chunks) at a time, one id per lane.
  int issued = 0;
  int ids = -1;  // this lane's block id for page 32 * (c / 4) + lane
  auto produce = [&](int c) -> bool {
    const int st = c % C::kStages;
    if ((c & 3) == 0) {
      const int lp = c * C::kPages + lane;
      ids = -1;
      if (lp < npages) {
        const int id = bt[page_lo + lp];
        ids = (id >= 0 && id < a.num_blocks) ? id : -1;
      }
    }
    if (c >= C::kStages && !wait_bar(bars.empty(st), ((c / C::kStages) - 1) & 1, abort_flag)) return false;
    uint32_t bytes = 0;
    int blk[C::kPages];
#pragma unroll
    for (int p = 0; p < C::kPages; ++p) {
      blk[p] = __shfl_sync(kFull, ids, (c & 3) * C::kPages + p);
      bytes += blk[p] >= 0 ? (uint32_t)L::kPage : 0u;
    }
    if (lane == 0) {
#pragma unroll
      for (int p = 0; p < C::kPages; ++p) pvalid[st * 8 + p] = blk[p] >= 0 ? 1 : 0;
      mbar_arrive_expect_tx(bars.full(st), bytes);
#pragma unroll
      for (int p = 0; p < C::kPages; ++p) {
        if (blk[p] >= 0) {
          const long page = (long)blk[p] * a.Hk + kvh;
          const uint8_t* src = a.cache + page * L::kPage;
          const uint32_t dst = sbase + C::kRing + st * C::kStageBytes;
          if constexpr (PRESET == 0) {
            tma_load_3d(dst + p * C::kKeyBlock, &tmap_keys, 0, 0, (int)page, bars.full(st));
            bulk_g2s(dst + C::kRestOff + p * C::kRestBytes, src + C::kKeyBlock, C::kRestBytes, bars.full(st));
          } else {
            bulk_g2s(dst + p * L::kPage, src, L::kPage, bars.full(st));
          }
        }
      }
    }
    issued = c + 1;
    return true;
  };
  if (warp == 0) {  // start streaming before the query prologue
    for (int c = 0; c < min(nchunks, 2); ++c) produce(c);
  }

  // ---- query rows (workers) and code-pair table (warps 2-3)
  if (tid >= 128) {
    // Q rows r = n * group + jq (zero beyond R) into the K-major, 128B-swizzled
    // B operand: row r, coordinate d at block d/64, line r, 16-byte chunk
    // ((d % 64) / 8) ^ (r % 8).  Eight threads per row, 16 coordinates each;
    // k3v4_nc rotates the rows: q_rot = H q / sqrt(128).
    const int r = (tid - 128) >> 3, part = (tid - 128) & 7;
    float x[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = 0.f;
    if (r < a.R) {
      const int n = r / a.group, jq = r % a.group;
      const uint4* qp = reinterpret_cast<const uint4*>(
          a.q + (((long)n * a.B + b) * a.Hq + kvh * a.group + jq) * kD + 16 * part);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint4 v4 = qp[u];
        const uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 h2 = *reinterpret_cast<const __half2*>(&w[e]);
          x[8 * u + 2 * e] = __low2float(h2);
          x[8 * u + 2 * e + 1] = __high2float(h2);
        }
      }
    }
    if (PRESET == 1) {
#pragma unroll
      for (int hs = 1; hs < 16; hs <<= 1)
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (!(e & hs)) {
            const float u = x[e], v = x[e + hs];
            x[e] = u + v;
            x[e + hs] = u - v;
          }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {  // strides 16, 32, 64: partner thread part ^ o
        const bool upper = (part & o) != 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float pv = __shfl_xor_sync(kFull, x[e], o);
          x[e] = upper ? pv - x[e] : x[e] + pv;
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] *= 0.08838834764831845f;
    }
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      const int d0 = 16 * part + 8 * hc;  // first coordinate of this 16-byte chunk
      uint8_t* rowp = sm + C::kQ + (d0 >> 6) * (NMMA * 128) + (r >> 3) * 1024 + (r & 7) * 128;
      const int chunk16 = (d0 & 63) >> 3;
      *reinterpret_cast<uint4*>(rowp + ((chunk16 ^ (r & 7)) << 4)) =
          make_uint4(pack_half2(x[8 * hc + 0], x[8 * hc + 1]), pack_half2(x[8 * hc + 2], x[8 * hc + 3]),
                     pack_half2(x[8 * hc + 4], x[8 * hc + 5]), pack_half2(x[8 * hc + 6], x[8 * hc + 7]));
    }
  } else if (PRESET == 1 && tid >= 64) {
    for (int i = tid - 64; i < 64 * 32; i += 64) {
      const int e = i >> 5;
      pairs[i] = (uint32_t)a.cb.c[e & 7] | ((uint32_t)a.cb.c[e >> 3] << 16);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float sl2 = kLog2e * 0.08838834764831845f;  // log2(e) / sqrt(128)

  if (warp < 4) {
    regs_dec<C::kRegCtl>();
    if (warp == 0) {
      // ================= producer: 8 pages per chunk into the ring
      for (int c = issued; c < nchunks; ++c)
        if (!produce(c)) break;
      // drain: copies still in flight must land before the CTA can exit
      for (int c = max(0, issued - C::kStages); c < issued; ++c)
        wait_bar(bars.full(c % C::kStages), (c / C::kStages) & 1, abort_flag, false);
    } else if (warp == 1 && lane == 0) {
      // ================= MMA issuer: S^T(c) as soon as chunk c's operands are in,
      // O^T += V^T P'^T for chunk c - 1 once its probabilities are
      constexpr uint32_t id_qk = idesc_f16(128, NMMA, 0, 0);
      constexpr uint32_t id_pv = idesc_f16(128, NMMA, 0, 1);
      int last_qk = -1, last_pv = -1;
      auto issue_pv = [&](int cc) -> bool {
        const int bb = cc & 1;
        if (!wait_bar(bars.pfull(bb), (cc >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = smem_desc(sbase + C::kP + bb * C::kPBytes + kk * 16 * C::kLine, 16, 8 * C::kLine,
                                        C::kSwzMode);
          mma_ts(tmem + C::kTO, tmem + C::kTAV + 64 * (cc % 3) + 8 * kk, bd, id_pv, (cc > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bars.pv(bb));
        last_pv = cc;
        return true;
      };
      bool ok = true;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int bb = c & 1;
        if (!wait_bar(bars.akv(bb), (c >> 1) & 1, abort_flag)) break;
        if (c >= 2 && !wait_bar(bars.sfree(bb), ((c - 2) >> 1) & 1, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = smem_desc(sbase + C::kQ + (kk >> 2) * (NMMA * 128) + (kk & 3) * 32, 16, 1024, 2);
          mma_ts(tmem + C::kTS + NMMA * bb, tmem + C::kTAK + 64 * bb + 8 * kk, bd, id_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bars.qk(bb));
        last_qk = c;
        if (c >= 1) ok = issue_pv(c - 1);
      }
      if (ok && last_qk == nchunks - 1 && nchunks > 0) issue_pv(nchunks - 1);
      // drain the MMAs this thread issued before tensor memory is freed
      if (last_qk >= 0) wait_bar(bars.qk(last_qk & 1), (last_qk >> 1) & 1, abort_flag, false);
      if (last_pv >= 0) wait_bar(bars.pv(last_pv & 1), (last_pv >> 1) & 1, abort_flag, false);
    }
  } else {
    if constexpr (C::kW > 1) regs_inc<C::kRegW>();
    // ================= workers: thread t = TMEM lane t (token t / coordinate t)
    const int wg = (warp - 4) >> 2;  // worker warpgroup
    const int sw = warp & 3;
    const int t = sw * 32 + lane;
    const uint32_t lane_q = (uint32_t)(sw * 32) << 16;
    const uint32_t bar_id = 1 + wg;
    const int pg_t = t >> 4, off_t = t & 15;  // token t of a chunk: page and row
    // running maxima start at a finite floor: a masked score (-inf) then always
    // gives p = 2^-inf = 0, and the first visible score forces a rescale
    constexpr float kFloor = -1.0e30f;
    float m[kNC], l[kNC], zs[kNC];
#pragma unroll
    for (int r = 0; r < kNC; ++r) {
      m[r] = kFloor;
      l[r] = 0.f;
      zs[r] = 0.f;
    }
    bool aborted = false;
    for (int it = 0; it <= nchunks; ++it) {
      // ---------- part A: this warpgroup's share of chunk `it`'s operands
      if (it < nchunks && !aborted) {
        const int c = it, st = c % C::kStages, bb = c & 1;
        bool ok = wait_bar(bars.full(st), (c / C::kStages) & 1, abort_flag);
        if (ok && c >= 2) ok = wait_bar(bars.qk(bb), ((c - 2) >> 1) & 1, abort_flag);  // A_K[c % 2] read by S^T(c - 2)
        // token params [c % 3] read by softmax(c - 3) before its sfree; softmax(c - 1)
        // on the same barrier cannot finish before this warpgroup's part B of it
        if (ok && c >= 3 && wg == 0) ok = wait_bar(bars.sfree((c - 3) & 1), ((c - 3) >> 1) & 1, abort_flag);
        // A_V[c % 3] read by O^T(c - 3); O^T(c - 1), on the same barrier, is not
        // issued before every worker has finished this part, so the parity is unambiguous
        if (ok && c >= 3) ok = wait_bar(bars.pv((c - 3) & 1), ((c - 3) >> 1) & 1, abort_flag);
        if (!ok) {
          aborted = true;
        } else {
          const uint8_t* stage = sm + C::kRing + st * C::kStageBytes;
          // page p's fields at pgf(p) + L::kVal / kScale / kZero / kNc
          auto pgf = [&](int p) -> const uint8_t* {
            return PRESET == 0 ? stage + C::kRestOff + p * C::kRestBytes - C::kKeyBlock : stage + p * L::kPage;
          };
          // keys of token t, coordinates [2 kKC wg, 2 kKC wg + 2 kKC) -> A_K[bb], lane t
          {
            uint32_t r[kKC];
            if constexpr (PRESET == 0) {
              // row off_t of page pg_t's key block: 16-byte chunk q sits at q ^ (off_t % 8)
              const uint8_t* kr = stage + pg_t * C::kKeyBlock + off_t * kD;
#pragma unroll
              for (int q = 0; q < kKC / 8; ++q) {
                const int qq = (kKC / 8) * wg + q;  // logical 16-byte chunk of the row
                const uint4 w = *reinterpret_cast<const uint4*>(kr + ((qq ^ (off_t & 7)) << 4));
                r[8 * q + 0] = e4m3x2_to_half2(w.x);
                r[8 * q + 1] = e4m3x2_to_half2(w.x >> 16);
                r[8 * q + 2] = e4m3x2_to_half2(w.y);
                r[8 * q + 3] = e4m3x2_to_half2(w.y >> 16);
                r[8 * q + 4] = e4m3x2_to_half2(w.z);
                r[8 * q + 5] = e4m3x2_to_half2(w.z >> 16);
                r[8 * q + 6] = e4m3x2_to_half2(w.w);
                r[8 * q + 7] = e4m3x2_to_half2(w.w >> 16);
              }
            } else {
              // 3-bit codes of coordinates [2 kKC wg, ...) start at byte 6 kKC wg / 8
              constexpr int kWords = 6 * kKC / 32;
              const uint32_t* kw = reinterpret_cast<const uint32_t*>(stage + pg_t * L::kPage + L::kKey + off_t * 48 +
                                                                     (6 * kKC / 8) * wg);
              uint32_t wd[kWords + 1];
#pragma unroll
              for (int u = 0; u < kWords; ++u) wd[u] = kw[u];
              wd[kWords] = 0u;
#pragma unroll
              for (int jj = 0; jj < kKC; ++jj) {  // pair jj: codes of 2jj, 2jj+1 at bits 6jj .. 6jj+5
                const int bit = 6 * jj, wi = bit >> 5, sh = bit & 31;
                uint32_t f = wd[wi] >> sh;
                if (sh > 26) f |= wd[wi + 1] << (32 - sh);
                r[jj] = pairs[(f & 63u) * 32 + lane];
              }
            }
            tmem_st_cols<kKC>(tmem + lane_q + C::kTAK + 64 * bb + kKC * wg, r);
          }
          // value codes of coordinate t, tokens [2 kKC wg, ...) = pages [kKC wg / 8, ...) -> A_V[bb]
          {
            uint32_t r[kKC];
#pragma unroll
            for (int pp = 0; pp < kKC / 8; ++pp) {
              const int p = (kKC / 8) * wg + pp;
              const uint2 w = *reinterpret_cast<const uint2*>(pgf(p) + L::kVal + 8 * t);
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const uint32_t x = half ? w.y : w.x;  // 4 bytes: token pairs of this coordinate
                const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint32_t y = __byte_perm(lo, hi, (uint32_t)k | ((uint32_t)(4 + k) << 8));
                  r[8 * pp + 4 * half + k] = y & 0x000F000Fu;  // fp16 bits = code: code * 2^-24
                }
              }
            }
            tmem_st_cols<kKC>(tmem + lane_q + C::kTAV + 64 * (c % 3) + kKC * wg, r);
          }
          // per-token parameters of token t (warpgroup 0)
          if (wg == 0) {
            const int pos = (page_lo + c * C::kPages) * kBlock + t;
            const bool valid = pvalid[st * 8 + pg_t] != 0 && pos < t_hi;
            float cs = sl2, sv = 0.f, zv = 0.f;
            int rmin = 1 << 20;
            if (valid) {
              const uint8_t* pg = pgf(pg_t);
              if constexpr (PRESET == 1)
                cs = __half2float(*reinterpret_cast<const __half*>(pg + L::kNc + 2 * off_t)) * sl2;
              sv = __half2float(*reinterpret_cast<const __half*>(pg + L::kScale + 2 * off_t));
              zv = __half2float(*reinterpret_cast<const __half*>(pg + L::kZero + 2 * off_t));
              rmin = 0;
              if (a.causal) {
                const int nmin = pos - L_b + a.n_spec;  // draft n sees this token iff n >= nmin
                rmin = nmin <= 0 ? 0 : nmin * a.group;
              }
            }
            colp[(c % 3) * 128 + t] = make_float4(cs, sv, zv, __int_as_float(rmin));
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bars.akv(bb));
            mbar_arrive(bars.empty(st));
          }
        }
      }
      // ---------- part B: softmax of chunk it - 1 for rows [16 wg, 16 wg + 16)
      if (it >= 1) {
        const int c = it - 1, bb = c & 1;
        const bool ok = !aborted && wait_bar(bars.qk(bb), (c >> 1) & 1, abort_flag) &&
                        wait_bar(bars.akv(bb), (c >> 1) & 1, abort_flag);
        // leave the loop together: the named barriers below need all four warps
        if (bar_red_or(bar_id, 128, !ok || aborted)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const float4 cp = colp[(c % 3) * 128 + t];
        const int rmin = __float_as_int(cp.w);
        const uint32_t s_addr = tmem + lane_q + C::kTS + NMMA * bb + kNC * wg;
        float y[kNC];
        auto load_scores = [&]() {
          uint32_t r[kNC];
          tmem_ld<kNC>(s_addr, r);
          tc_wait_ld();
          if (__all_sync(kFull, rmin <= kNC * wg)) {  // every row of this warpgroup sees these tokens
#pragma unroll
            for (int k = 0; k < kNC; ++k) y[k] = __uint_as_float(r[k]) * cp.x;
          } else {
#pragma unroll
            for (int k = 0; k < kNC; ++k)
              y[k] = (kNC * wg + k < rmin) ? -CUDART_INF_F : __uint_as_float(r[k]) * cp.x;
          }
        };
        load_scores();
        bool need = false;
#pragma unroll
        for (int k = 0; k < kNC; ++k) need |= y[k] > m[k] + kRescaleThreshold;
        need = bar_red_or(bar_id, 128, need);
        if (need) {
          // exact maximum of this chunk for each row over the 128 tokens
          // (reduces y in place; the scores are reloaded from tensor memory)
          warp_transpose_reduce<kNC, true>(y, lane);
          float* rmax = red + (wg * 3 + 0) * 4 * kNC;
          if (lane < kNC) rmax[sw * kNC + lane] = y[0];
          named_bar(bar_id, 128);
#pragma unroll
          for (int k = 0; k < kNC; ++k)
            y[k] = fmaxf(fmaxf(rmax[k], rmax[kNC + k]), fmaxf(rmax[2 * kNC + k], rmax[3 * kNC + k]));
          bool change = false;
#pragma unroll
          for (int k = 0; k < kNC; ++k) change |= y[k] > m[k];
          const bool rescale_o = change && c > 0;  // uniform across the warpgroup
          if (rescale_o) {
            // O^T holds chunks < c: rescale it after the previous P.V has landed
            // and before this chunk's is issued
            if (!wait_bar(bars.pv((c - 1) & 1), ((c - 1) >> 1) & 1, abort_flag)) aborted = true;
            tc_fence_after();
          }
          uint32_t r[kNC];
          const uint32_t o_addr = tmem + lane_q + C::kTO + kNC * wg;
          if (rescale_o) {
            tmem_ld<kNC>(o_addr, r);
            tc_wait_ld();
          }
#pragma unroll
          for (int k = 0; k < kNC; ++k) {
            const float mn = fmaxf(m[k], y[k]);
            const float al = ex2(m[k] - mn);
            m[k] = mn;
            l[k] *= al;
            zs[k] *= al;
            r[k] = __float_as_uint(__uint_as_float(r[k]) * al);
          }
          if (rescale_o) {
            tmem_st<kNC>(o_addr, r);
            tc_wait_st();
          }
          load_scores();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sfree(bb));
        if (c >= 2 && !wait_bar(bars.pv(bb), ((c - 2) >> 1) & 1, abort_flag)) aborted = true;
        // probabilities, row sums, zero term; P' = p * scale into the MN-major B tile
        uint8_t* pbuf = sm + C::kP + bb * C::kPBytes;
#pragma unroll
        for (int q = 0; q < kNC / 8; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 8 * q + 2 * e;
            const float p0 = ex2(y[k] - m[k]);
            const float p1 = ex2(y[k + 1] - m[k + 1]);
            l[k] += p0;
            l[k + 1] += p1;
            zs[k] = fmaf(p0, cp.z, zs[k]);
            zs[k + 1] = fmaf(p1, cp.z, zs[k + 1]);
            pk[e] = pack_half2(p0 * cp.y, p1 * cp.y);
          }
          const uint32_t lg = (uint32_t)((t >> 3) * (8 * C::kLine) + (t & 7) * C::kLine + wg * kNC * 2 + 16 * q);
          const uint32_t ph = lg ^ (((lg >> 7) & ((1u << C::kSwzBits) - 1u)) << 4);
          *reinterpret_cast<uint4*>(pbuf + ph) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.pfull(bb));
      }
    }
    // ---- epilogue: l and zero term over all 128 tokens, then O^T / l
    {
      float v[kNC];
#pragma unroll
      for (int k = 0; k < kNC; ++k) v[k] = l[k];
      warp_transpose_reduce<kNC, false>(v, lane);
      float* rl = red + (wg * 3 + 1) * 4 * kNC;
      if (lane < kNC) rl[sw * kNC + lane] = v[0];
#pragma unroll
      for (int k = 0; k < kNC; ++k) v[k] = zs[k];
      warp_transpose_reduce<kNC, false>(v, lane);
      float* rz = red + (wg * 3 + 2) * 4 * kNC;
      if (lane < kNC) rz[sw * kNC + lane] = v[0];
    }
    named_bar(bar_id, 128);
    uint32_t o[kNC];
#pragma unroll
    for (int k = 0; k < kNC; ++k) o[k] = 0u;
    if (nchunks > 0 && !aborted) {
      const int lc = nchunks - 1;
      if (wait_bar(bars.pv(lc & 1), (lc >> 1) & 1, abort_flag)) {
        tc_fence_after();
        tmem_ld<kNC>(tmem + lane_q + C::kTO + kNC * wg, o);
        tc_wait_ld();
      } else {
        aborted = true;
      }
    }
    aborted = aborted || (*abort_flag != 0u);
    // per-row constants (threads 0..15): 1 / l, zero term / l, log-sum-exp
    float* rowc = red + C::kW * 3 * 4 * kNC + wg * 2 * kNC;
    if (t < kNC) {
      const float* rl = red + (wg * 3 + 1) * 4 * kNC;
      const float* rz = red + (wg * 3 + 2) * 4 * kNC;
      const float lt = (rl[t] + rl[kNC + t]) + (rl[2 * kNC + t] + rl[3 * kNC + t]);
      const float zt = (rz[t] + rz[kNC + t]) + (rz[2 * kNC + t] + rz[3 * kNC + t]);
      float mt = m[0];
#pragma unroll
      for (int k = 1; k < kNC; ++k) mt = (t == k) ? m[k] : mt;
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      rowc[t] = inv * 16777216.0f;  // O^T holds the value codes as fp16 subnormals (code * 2^-24)
      rowc[kNC + t] = zt * inv;
      const int row = kNC * wg + t;
      if (row < a.R) {
        const long orow = (((long)(row / a.group) * a.B + b) * a.Hq + kvh * a.group + row % a.group) * a.S + split;
        a.part_lse[orow] = aborted ? CUDART_NAN_F : (lt > 0.f ? (mt + log2f(lt)) * kLn2 : -CUDART_INF_F);
      }
    }
    named_bar(bar_id, 128);
    // rows 16 wg + k = n * group + j, walked incrementally
    int jj = (kNC * wg) % a.group;
    float* po = a.part_o + ((((long)((kNC * wg) / a.group) * a.B + b) * a.Hq + kvh * a.group + jj) * a.S + split) * kD + t;
    const long step_j = (long)a.S * kD, step_n = ((long)a.B * a.Hq - a.group) * a.S * kD;
#pragma unroll
    for (int k = 0; k < kNC; ++k) {
      if (kNC * wg + k < a.R) *po = aborted ? CUDART_NAN_F : fmaf(__uint_as_float(o[k]), rowc[k], rowc[kNC + k]);
      po += step_j;
      if (++jj == a.group) {
        jj = 0;
        po += step_n;
      }
    }
  }

  // ---- teardown: every role has drained its asynchronous work
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// k8v4 key blocks as a 3-D byte tensor {128 bytes, 16 tokens, pages} with the
// page stride of the cache; one box = one page's keys, 128B-swizzled in smem
cudaError_t make_key_map(const VerifyArgs& a, CUtensorMap* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t pages = (cuuint64_t)a.num_blocks * (cuuint64_t)a.Hk;
  cuuint64_t gdim[3] = {128, 16, pages > 0 ? pages : 1};
  cuuint64_t gstride[2] = {128, (cuuint64_t)K8::kPage};
  cuuint32_t box[3] = {128, 16, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.cache), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int PRESET, int NMMA>
cudaError_t launch_tc(const VerifyArgs& a, cudaStream_t st) {
  using C = Cfg<PRESET, NMMA>;
  auto kern = verify_stage1_tc_kernel<PRESET, NMMA>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    // setmaxnreg.inc waits for registers released by other warps of the CTA:
    // refuse to launch if the compiled register count cannot cover the split
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * C::kThreads < C::kRegNeeded) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  if (PRESET == 0) {
    e = make_key_map(a, &tmap);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(a.S, a.Hk, a.B);
  kern<<<grid, C::kThreads, C::kSmem, st>>>(a, tmap);
  return cudaGetLastError();
}

}  // namespace

bool verify_stage1_tc_supported(const VerifyArgs& a) { return a.R <= 64; }

cudaError_t launch_verify_stage1_tc(int preset, const VerifyArgs& a, cudaStream_t st) {
  if (preset == 0) {
    if (a.R <= 16) return launch_tc<0, 16>(a, st);
    if (a.R <= 32) return launch_tc<0, 32>(a, st);
    return launch_tc<0, 64>(a, st);
  }
  if (a.R <= 16) return launch_tc<1, 16>(a, st);
  if (a.R <= 32) return launch_tc<1, 32>(a, st);
  return launch_tc<1, 64>(a, st);
}

cudaError_t read_device_error(unsigned int* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tq_device_error, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tq_device_error, &zero, sizeof(unsigned int));
}

}  // namespace tq
