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
// with A operands in tensor memory (written with tcgen05.st) and B operands
// in shared memory (Q once per CTA; P' per chunk).
//   keys   : k8v4 e4m3 -> f16 exactly (the key block of a page arrives by TMA
//            with 128-byte swizzle, so the per-token row reads are free of
//            bank conflicts); k3v4_nc 3-bit code pairs -> fp16 centroid pairs
//            through a per-lane replicated table; the norm correction nc_t
//            scales token t's scores after the MMA; the query is rotated
//            once, q_rot = H q / sqrt(D).
//   values : a 4-bit code c enters the MMA as the fp16 subnormal c * 2^-24
//            (even tokens) or 16 c * 2^-24 (odd tokens, whose probability is
//            divided by 16), so that one 32-bit word of eight codes becomes
//            four f16x2 operand words with one shift and four masks; the
//            factor 2^24 is undone on the output.  P' = p * scale_t; the zero
//            term sum_t p_t zero_t and l = sum_t p_t are kept per thread in
//            fp32 and reduced at the end.
// Softmax: thread t owns token t (its S^T lane) and up to 32 query rows.  The
// running maximum is updated lazily: only when some score exceeds it by more
// than 8 (log2 units) is the exact chunk maximum computed across the 128
// tokens and O^T, l and the zero term rescaled; otherwise probabilities stay
// bounded by 2^8 and the stale maximum is used (any reference point gives the
// same softmax).
//
// Warp roles with 64 rows: warps 0, 2, 3 = producers (block ids + copies),
// warp 1 = MMA issuer and TMEM owner; warpgroup 1 dequantises chunk c (A_K[c %
// 2], A_V[c % 3] and the per-token parameters) while softmax warpgroup j (rows
// [32 j, 32 j + 32)) works on an earlier chunk.  With up to 32 rows: warps 2, 3
// = producers, warp 1 issues the S^T MMAs (and owns TMEM), warp 0 the P.V
// MMAs, and softmax warpgroup j takes every row of chunks j, j + 2, ... (two
// streams merged by log-sum-exp at the end).  Every wait on an mbarrier is
// bounded: on expiry the CTA sets an abort flag and the sticky device error
// word, drains its in-flight copies and MMAs, frees its tensor memory and
// writes NaN partials.
#include <math_constants.h>

#include <atomic>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "store_ops.cuh"
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
// the cross-CTA waits of the single-launch verify give up after kSpinNs of
// polling (or kSpinTries polls, should the timer not advance)
constexpr uint64_t kSpinNs = 500000000ull;
constexpr uint32_t kSpinTries = 1u << 24;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int PRESET, int NR>
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
  static constexpr int kStages = PRESET == 0 ? 5 : PRESET == 4 ? 6 : 8;
  static constexpr int kKeyBits = key_bits<PRESET>();  // 0: FP8 keys
  // code-pair table: entry e = (code of coordinate 2j) | (code of 2j+1) << bits,
  // replicated for the 32 lanes
  static constexpr int kPairEntries = PRESET == 0 ? 0 : 1 << (2 * kKeyBits);
  // two softmax warpgroups: with 64 rows each takes 32 rows of every chunk;
  // with up to 32 rows each takes every row of alternate chunks (two
  // streams, each with its own S^T buffers, O^T accumulator and running
  // maximum, merged by log-sum-exp in the epilogue)
  static constexpr int kSW = 2;
  static constexpr int kStreams = NR == 64 ? 1 : 2;
  static constexpr int kRS = NR == 64 ? 32 : NR;  // query rows per softmax thread
  static constexpr int kSbuf = 2 * kStreams;      // S^T buffers
  // token-parameter slots (chunk c: c % kColP): a slot is rewritten kSbuf + 2
  // chunks on when the softmax reads chunk c's parameters before it releases
  // S^T(c) (two streams), kSbuf + 4 when it reads them after (64 rows)
  static constexpr int kColP = kStreams == 2 ? 8 : kSbuf + 4;
  static constexpr int kThreads = 256 + 128 * kSW;
  // per-thread register budgets after setmaxnreg (control / dequant /
  // softmax); their sum must stay within what the launch granted (checked at
  // launch: 128 registers a thread for 512 threads, 168 for 384)
  // (setmaxnreg is executed by all four warps of a warpgroup together)
  static constexpr int kRegCtl = 48;
  static constexpr int kRegDq = 96;
  static constexpr int kRegSm = 184;
  static constexpr int kRegNeeded = 128 * kRegCtl + 128 * kRegDq + 128 * kSW * kRegSm;
  static_assert(kRegNeeded <= 65536, "register split exceeds the register file");
  static constexpr int kLine = 2 * NR;  // bytes of one P' line (one token)
  static constexpr int kSwzBits = NR == 64 ? 3 : (NR == 32 ? 2 : 1);
  static constexpr uint32_t kSwzMode = NR == 64 ? 2u : (NR == 32 ? 4u : 6u);
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kRing = 0;
  static constexpr int kQ = align_up(kStages * kStageBytes, 1024);
  static constexpr int kQBytes = 2 * NR * 128;  // K-major, 128B swizzle, 2 x 64-coordinate blocks
  static constexpr int kP = kQ + align_up(kQBytes, 1024);
  static constexpr int kPBytes = kTok * kLine;  // one buffer
  static constexpr int kCol = kP + 3 * kPBytes;  // float4 [kColP][128]: score scale, P' scale, v zero, first row
  // per softmax warpgroup (floats): -m [32] @0, rescale factors [32] @32,
  // row constants float2 [32] @64, per-warp row maxima [4][32] @128, per-warp
  // row sums of l and of the zero term [2][128] @256, rows without a maximum
  // yet (bit mask) @512
  static constexpr int kRed = kCol + kColP * kTok * 16;
  static constexpr int kRedWG = 4096;
  static constexpr int kPair = kRed + kSW * kRedWG;  // u32 [kPairEntries][32] (coded keys)
  static constexpr int kPValid = kPair + kPairEntries * 32 * 4;  // u8 [kStages][8]
  static constexpr int kBar = align_up(kPValid + kStages * 8, 8);
  // full[kStages] empty[kStages] ak[4] pfull[3] pv[3] av[3] pvs[2]
  // sready[kSbuf] sfree[kSbuf]
  // producers: warps 0, 2, 3 copy pages 0-2, 3-5, 6-7 of a chunk (64 rows,
  // one MMA issuer); warps 2, 3 copy pages 0-3, 4-7 (two streams: warp 0
  // issues the P.V MMAs)
  static constexpr int kProducers = kStreams == 2 ? 2 : 3;
  static constexpr int kNumBars = 2 * kStages + 15 + 2 * kSbuf;
  static constexpr int kMisc = kBar + 8 * kNumBars;  // u32 tmem base, u32 abort, u32 merge go
  static constexpr int kSmem = kMisc + 16 + 1024;    // + alignment slack
  // tensor memory columns
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTAK = 0;    // A_K[2]: 64 cols each (token lanes, coordinate pairs)
  static constexpr uint32_t kTAV = 128;  // A_V[3]: 64 cols each (coordinate lanes, token pairs)
  static constexpr uint32_t kTS = 320;   // S^T[kSbuf]: NR cols each
  static constexpr uint32_t kTO = 320 + kSbuf * NR;  // O^T[kStreams]: NR cols each
  static_assert(kTO + kStreams * NR <= kTmemCols, "tensor memory overflow");
  static_assert(kSmem <= 227 * 1024, "shared memory overflow");
};

// Barriers.  Each ring is deep enough that no arrival for chunk c + depth can
// complete before every waiter for chunk c has waited: a waiter never sees a
// barrier two phases ahead of the one it waits for.  (ak: keys of chunk c + 4
// need S^T(c + 2) done, issued after softmax(c) released S^T(c), which it
// does after its own wait on ak(c).)
struct Bars {
  uint32_t base;
  int stages;
  int sbuf;  // S^T buffers
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (stages + s); }
  __device__ uint32_t ak(int i) const { return base + 8 * (2 * stages + i); }         // A_K + token params (c % 4)
  __device__ uint32_t pfull(int i) const { return base + 8 * (2 * stages + 4 + i); }  // P' written (c % 3)
  __device__ uint32_t pv(int i) const { return base + 8 * (2 * stages + 7 + i); }     // O^T += V^T P'^T done (c % 3)
  __device__ uint32_t av(int i) const { return base + 8 * (2 * stages + 10 + i); }    // A_V written (c % 3)
  // P.V(c) done, per stream (c % 2; two-stream mode only)
  __device__ uint32_t pvs(int j) const { return base + 8 * (2 * stages + 13 + j); }
  // S^T = K Q^T done and chunk c's parameters written (c % sbuf): four
  // dequant arrivals plus the issuer's commit, which also covers every
  // earlier P.V
  __device__ uint32_t sready(int b) const { return base + 8 * (2 * stages + 15 + b); }
  __device__ uint32_t sfree(int b) const { return base + 8 * (2 * stages + 15 + sbuf + b); }  // S^T(c) read (c % sbuf)
};

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for a global counter written by other CTAs of the same
// (cooperative, hence co-resident) grid to reach target; false when it
// expired (after kSpinNs), which is recorded in the device error word.
__device__ __forceinline__ bool spin_until_at_least(const uint32_t* counter, uint32_t target) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if ((i & 63) == 0) {
      const uint64_t t = now_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kSpinNs || i >= kSpinTries) break;
    }
    if (i >= 256) __nanosleep(64);
  }
  atomicOr(&g_tq_device_error, 1u);
  return false;
}

// Bounded wait by polling (the MMA issuers: no suspension between polls);
// false when the CTA aborted or this wait expired (which aborts).
__device__ __forceinline__ bool poll_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((i & 63) == 63) {
      const uint64_t t = now_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kSpinNs || i >= (1u << 28)) {
        *abort = 1u;
        atomicOr(&g_tq_device_error, 1u);
        return false;
      }
    }
  }
}

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

// two e4m3 codes (low and high byte) -> two f16 (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16) {
  uint32_t r;
  const uint16_t h = (uint16_t)(w16 & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

// 2^x, hardware approximation (relative error ~2^-22), -inf -> 0
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (2^lo, 2^hi) as an f16x2 pair from two fp32 exponents: one MUFU operation
// for two values (relative error ~2^-10); -inf -> 0
__device__ __forceinline__ uint32_t ex2_h2(float lo, float hi) {
  uint32_t h, y;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(h));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
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

// Position of chunk token t on the K axis of the P.V contraction.  Within
// each group of 8 tokens the value operand holds the pairs (0,5) (1,4) (2,7)
// (3,6), the order the nibble masks produce.
__device__ __forceinline__ int kappa(int t) {
  constexpr uint32_t kPos = 0x57136420u;  // nibble k: position of token k of a group
  return (t & ~7) | (int)((kPos >> (4 * (t & 7))) & 7u);
}

// FUSED: stage 2 in the same launch, a cooperative grid (every CTA
// resident).  The S splits of a (sequence, kv-head) write their partial rows
// into the scratch partials ([B][Hk][S][R] layout, a CTA's rows contiguous),
// count themselves in on the pair's arrival counter and wait for all S; split
// s then merges rows [s r, (s + 1) r) (r = ceil(R / S)) into the output.  The
// last split to finish its merge sets both counters back to zero.
template <int PRESET, int NR, bool FUSED>
__global__ void __launch_bounds__(Cfg<PRESET, NR>::kThreads, 1)
    verify_stage1_tc_kernel(VerifyArgs a, const __grid_constant__ CUtensorMap tmap_keys) {
  using C = Cfg<PRESET, NR>;
  using L = typename C::L;
  constexpr int kRS = C::kRS;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  uint8_t* pvalid = sm + C::kPValid;
  float4* colp = reinterpret_cast<float4*>(sm + C::kCol);
  uint32_t* pairs = reinterpret_cast<uint32_t*>(sm + C::kPair);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + C::kMisc + 4);
  const Bars bars{sbase + C::kBar, C::kStages, C::kSbuf};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // rows beyond 64 per kv-head are tiled across CTAs: this CTA takes rows
  // [row_off, row_off + Rt) of its (split, kv-head, sequence); the tiles of
  // a split stream the same pages (L2 serves the repeats)
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z / a.rtiles, rt = blockIdx.z % a.rtiles;
  const int row_off = rt * NR, Rt = min(a.R - row_off, NR);
  const int unit = rt * a.S + split;  // this CTA among the S x rtiles of its pair
  // ---- set-up: barriers, tensor memory (warp 1, first thing: shared and
  // tensor memory only, so it overlaps the wait for the previous grid)
  if (tid == 32) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bars.full(s), C::kProducers);
      mbar_init(bars.empty(s), 4);
    }
    for (int i = 0; i < 4; ++i) mbar_init(bars.ak(i), 4);
    // a chunk's S^T and P' are handled by both softmax warpgroups (64 rows)
    // or by one (two streams)
    constexpr int kPerChunk = 4 * C::kSW / C::kStreams;
    for (int i = 0; i < 3; ++i) {
      mbar_init(bars.av(i), 4);
      mbar_init(bars.pv(i), 1);
      mbar_init(bars.pfull(i), kPerChunk);
    }
    for (int i = 0; i < 2; ++i) mbar_init(bars.pvs(i), 1);
    for (int i = 0; i < C::kSbuf; ++i) {
      mbar_init(bars.sready(i), 5);
      mbar_init(bars.sfree(i), kPerChunk);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();

  // ---- this thread's part of the query rows, requested before anything else
  // (it depends on nothing but the launch): set-up thread t = tid - 128 < 4 NR
  // takes row r = t / 4, coordinates [32 (t % 4), 32 (t % 4) + 32)
  const int q_item = tid - 128, q_r = q_item >> 2, q_part = q_item & 3;
  const bool q_mine = tid >= 128 && q_item < 4 * NR;
  uint4 qv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) qv[u] = make_uint4(0u, 0u, 0u, 0u);
  if (q_mine && q_r < Rt) {
    const int n = (row_off + q_r) / a.group, jq = (row_off + q_r) % a.group;
    const uint4* qp =
        reinterpret_cast<const uint4*>(a.q + (((long)n * a.B + b) * a.Hq + kvh * a.group + jq) * kD + 32 * q_part);
#pragma unroll
    for (int u = 0; u < 4; ++u) qv[u] = qp[u];
  }

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
  // single-launch store + verify: the drafts sit at [L_b - n_spec, L_b);
  // the S splits of the pair store them (split s: drafts n = s mod S, on
  // producer warp 3 while the first pages are on their way) and count them
  // on the pair's draft counter; a split whose range holds drafts copies the
  // chunks from c_draft on only once all n_spec are counted
  const bool drafts = FUSED && a.dk != nullptr;
  const int d_lo = max(max(L_b - a.n_spec, t_lo), 0);
  const bool reads_drafts = drafts && d_lo < t_hi;
  const int c_draft = reads_drafts ? (d_lo - t_lo) / (C::kPages * kBlock) : nchunks;
  uint32_t* pair_tickets = FUSED ? a.tickets + ((long)b * a.Hk + kvh) * 4 : nullptr;
  const int32_t* bt = a.block_table + (long)b * a.max_blocks;

  // Producers (C::kProducers: warps 0, 2, 3 or warps 2, 3): producer w copies
  // pages [w ppw, (w + 1) ppw) of each chunk, one page per lane, since a warp
  // issues its lanes' copies one after another and each costs tens of
  // cycles.  Block ids are fetched 32 pages (4 chunks) at a time, one id per
  // lane, a group ahead.
  constexpr int kPpw = (C::kPages + C::kProducers - 1) / C::kProducers;  // pages per producer
  const bool producer = warp == 2 || warp == 3 || (C::kProducers == 3 && warp == 0);
  const int pw = C::kProducers == 3 ? (warp == 0 ? 0 : warp - 1) : warp - 2;
  const int p_lo = kPpw * pw, p_hi = min(C::kPages, p_lo + kPpw);
  int ids = -1, ids_next = -1;  // this lane's block id for page 32 * (c / 4) + lane, and for the next group
  // raw ids (validated when the page is copied, so that nothing waits for
  // them before the set-up barrier)
  auto fetch_ids = [&](int c) -> int {
    const int lp = c * C::kPages + lane;
    return lp < npages ? bt[page_lo + lp] : -1;
  };
  // the cache pages are read once per call: evict them from L2 first
  const uint64_t pol = producer ? l2_evict_first() : 0ull;
  auto produce = [&](int c) {
    const int st = c % C::kStages;
    int mine = __shfl_sync(kFull, ids, (c & 3) * C::kPages + (lane & 7));
    mine = (mine >= 0 && mine < a.num_blocks) ? mine : -1;
    const bool my = lane >= p_lo && lane < p_hi;
    const uint32_t nvalid = __popc(__ballot_sync(kFull, my && mine >= 0));
    // page flags first: the arrive below releases them to the consumers
    if (my) pvalid[st * 8 + lane] = mine >= 0 ? 1 : 0;
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bars.full(st), nvalid * (uint32_t)L::kPage);
    __syncwarp();
    if (my && mine >= 0) {
      const uint32_t dst = sbase + C::kRing + st * C::kStageBytes;
      const long page = (long)mine * a.Hk + kvh;
      const uint8_t* src = a.cache + page * L::kPage;
      if constexpr (PRESET == 0) {
        tma_load_3d_hint(dst + lane * C::kKeyBlock, &tmap_keys, 0, 0, (int)page, bars.full(st), pol);
        bulk_g2s_hint(dst + C::kRestOff + lane * C::kRestBytes, src + C::kKeyBlock, C::kRestBytes, bars.full(st), pol);
      } else {
        bulk_g2s_hint(dst + lane * L::kPage, src, L::kPage, bars.full(st), pol);
      }
    }
    __syncwarp();
  };
  if (producer && nchunks > 0) {  // in flight during the set-up
    if (PRESET == 0 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_keys) : "memory");
    ids = fetch_ids(0);
    ids_next = fetch_ids(4);
  }

  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_bar();  // barriers initialised, tensor memory allocated
  tc_fence_after();

  // the whole ring goes out at once (up to the chunk holding drafts this
  // split stores first); the first chunk lands about as early as when it
  // is requested alone.  The producers go on to their loop without waiting
  // for the rest of the set-up.
  const int prefill = min(min(nchunks, C::kStages), min(c_draft, 4));
  if (producer)
    for (int c = 0; c < prefill; ++c) produce(c);

  // ---- query rows and code-pair table (dequant + softmax warpgroups); the
  // other warps that need them (MMA issuer) wait on named barrier 14
  if (tid >= 128) {
    // Q rows r = n * group + jq (zero beyond R) into the K-major, 128B-swizzled
    // B operand: row r, coordinate d at block d/64, line r, 16-byte chunk
    // ((d % 64) / 8) ^ (r % 8).  k3v4_nc rotates the rows:
    // q_rot = H diag(signs) q / sqrt(128).
    if (q_mine) {
      float x[32];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 h2 = *reinterpret_cast<const __half2*>(&w[e]);
          x[8 * u + 2 * e] = __low2float(h2);
          x[8 * u + 2 * e + 1] = __high2float(h2);
        }
      }
      if (PRESET != 0) {
        // signs of coordinates 32 part + e, then the butterflies of strides
        // 1 .. 16 in the thread and 32, 64 across the row's four threads
        const uint32_t sg = a.signs[q_part];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if ((sg >> e) & 1u) x[e] = -x[e];
#pragma unroll
        for (int hs = 1; hs < 32; hs <<= 1)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!(e & hs)) {
              const float u = x[e], v = x[e + hs];
              x[e] = u + v;
              x[e + hs] = u - v;
            }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {  // partner thread part ^ o
          const bool upper = (q_part & o) != 0;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float pv = __shfl_xor_sync(kFull, x[e], o);
            x[e] = upper ? pv - x[e] : x[e] + pv;
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] *= 0.08838834764831845f;
      }
#pragma unroll
      for (int hc = 0; hc < 4; ++hc) {
        const int d0 = 32 * q_part + 8 * hc;  // first coordinate of this 16-byte chunk
        uint8_t* rowp = sm + C::kQ + (d0 >> 6) * (NR * 128) + (q_r >> 3) * 1024 + (q_r & 7) * 128;
        const int chunk16 = (d0 & 63) >> 3;
        *reinterpret_cast<uint4*>(rowp + ((chunk16 ^ (q_r & 7)) << 4)) =
            make_uint4(pack_half2(x[8 * hc + 0], x[8 * hc + 1]), pack_half2(x[8 * hc + 2], x[8 * hc + 3]),
                       pack_half2(x[8 * hc + 4], x[8 * hc + 5]), pack_half2(x[8 * hc + 6], x[8 * hc + 7]));
      }
    }
    if (PRESET != 0) {
      constexpr int kB = C::kKeyBits, kLv = 1 << kB;
      for (int i = tid - 128; i < C::kPairEntries * 32; i += C::kThreads - 128) {
        const int e = i >> 5;
        pairs[i] = (uint32_t)a.cb.c[e & (kLv - 1)] | ((uint32_t)a.cb.c[e >> kB] << 16);
      }
    }
  }
  if (!producer) {
    fence_async_smem();
    named_bar(14, C::kThreads - 32 * C::kProducers);
  }
  const uint32_t tmem = *tmem_slot;
  const float sl2 = kLog2e * 0.08838834764831845f;  // log2(e) / sqrt(128)

  if (warp < 4) {
    regs_dec<C::kRegCtl>();
    if (producer) {
      if constexpr (FUSED) {
        if (warp == 3 && drafts) {
          // ================= the drafts n = split mod S of this pair, between
          // the first chunks' copies and the next ones (this warp's copies of
          // chunk prefill wait for a free ring stage anyway); skipped drafts
          // (no position, invalid block) count too
          uint32_t count = 0;
          for (int n = unit; n < a.n_spec; n += a.S * a.rtiles) {
            ++count;
            const int pos = L_b - a.n_spec + n;
            if (pos < 0) continue;
            const int id = a.block_table[(long)b * a.max_blocks + pos / kBlock];
            if (id < 0 || id >= a.num_blocks) continue;
            uint8_t* page = a.cache_w + ((long)id * a.Hk + kvh) * L::kPage;
            const long base = (((long)b * a.n_spec + n) * a.Hk + kvh) * kD + 4 * lane;
            const uint2 kr = *reinterpret_cast<const uint2*>(a.dk + base);
            const uint2 vr = *reinterpret_cast<const uint2*>(a.dv + base);
            const uint16_t kh[4] = {(uint16_t)(kr.x & 0xFFFF), (uint16_t)(kr.x >> 16), (uint16_t)(kr.y & 0xFFFF),
                                    (uint16_t)(kr.y >> 16)};
            const uint16_t vh[4] = {(uint16_t)(vr.x & 0xFFFF), (uint16_t)(vr.x >> 16), (uint16_t)(vr.y & 0xFFFF),
                                    (uint16_t)(vr.y >> 16)};
            store_ops::store_token<PRESET>(page, pos % kBlock, lane, kh, vh, a.cb, a.plain_norm != 0,
                                           store_ops::lane_signs(a.signs, lane));
          }
          if (count > 0) {
            // the pages' new bytes (generic proxy) are read next by bulk copies
            // of this or another CTA: proxy fence, then a release at gpu scope
            asm volatile("fence.proxy.async.global;\n" ::: "memory");
            __syncwarp();
            if (lane == 0)
              asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(pair_tickets + 2), "r"(count) : "memory");
          }
        }
      }
      // ================= producers: their pages of each chunk into the ring
      int c = prefill;
      for (; c < nchunks; ++c) {
        if ((c & 3) == 0 && c > 0) {  // group 0's ids are loaded before the set-up
          ids = ids_next;
          ids_next = fetch_ids(c + 4);  // lands while this group is copied
        }
        if (c >= C::kStages && !wait_bar(bars.empty(c % C::kStages), ((c / C::kStages) - 1) & 1, abort_flag)) break;
        if (c == c_draft) {
          // every draft of the pair is stored (by whichever split): the
          // generic-proxy writes of other CTAs, acquired here, precede the
          // bulk copies of this warp
          bool ok = true;
          if (lane == 0) ok = spin_until_at_least(pair_tickets + 2, (uint32_t)a.n_spec);
          ok = __shfl_sync(kFull, ok, 0);
          if (!ok) {
            *abort_flag = 1u;
            break;
          }
          asm volatile("fence.proxy.async.global;\n" ::: "memory");
        }
        produce(c);
      }
      // drain: copies still in flight must land before the CTA can exit
      for (int cc = max(0, c - C::kStages); cc < c; ++cc)
        wait_bar(bars.full(cc % C::kStages), (cc / C::kStages) & 1, abort_flag, false);
    } else if (C::kStreams == 2 || warp == 1) {
      constexpr uint32_t kL = C::kLine;  // P' line bytes: 16 lines per K-step
      constexpr uint32_t id_qk = idesc_f16(128, NR, 0, 0);
      constexpr uint32_t id_pv = idesc_f16(128, NR, 0, 1);
      constexpr uint32_t kQ1 = NR * 8;  // second 64-coordinate block of Q, in 16-byte units
      const uint64_t q_desc = smem_desc(sbase + C::kQ, 16, 1024, 2);
      const uint64_t p_desc = smem_desc(sbase + C::kP, 16, 8 * C::kLine, C::kSwzMode);
      // S^T(c) = K_hat(c) Q^T into S^T buffer c % kSbuf
      auto issue_qk = [&](int c) {
        tc_fence_after();
        mma_ts_x8<2, 4, 6, kQ1, kQ1 + 2, kQ1 + 4, kQ1 + 6>(tmem + C::kTS + NR * (c % C::kSbuf),
                                                           tmem + C::kTAK + 64 * (c & 1), q_desc, id_qk, 0u);
        tc_commit(bars.sready(c % C::kSbuf));
      };
      // O^T += V^T P'^T(c) into the O^T of the chunk's stream (a stream's first P.V overwrites it)
      auto issue_pv = [&](int c) {
        tc_fence_after();
        mma_ts_x8<kL, 2 * kL, 3 * kL, 4 * kL, 5 * kL, 6 * kL, 7 * kL>(
            tmem + C::kTO + NR * (c % C::kStreams), tmem + C::kTAV + 64 * (c % 3),
            p_desc + (uint64_t)(((c % 3) * C::kPBytes) >> 4), id_pv, c >= C::kStreams ? 1u : 0u);
        tc_commit(bars.pv(c % 3));
        if (C::kStreams == 2) tc_commit(bars.pvs(c & 1));
      };
      if constexpr (C::kStreams == 1) {
        // ================= MMA issuer (64 rows; warp 1, one thread), never
        // blocked on one operand while the other kind of MMA could go:
        // S^T(c) once softmax(c - 2) released its buffer and the keys of
        // chunk c are in tensor memory; P.V(c) once softmax(c) wrote P'(c)
        // and the values of chunk c are in tensor memory.  S^T(c) is issued
        // only after P.V(c - 3): a commit tracks every earlier MMA of this
        // thread, so the completion of S^T(c) then also means that P.V(c - 3)
        // is done, which frees P' buffer c % 3 and value buffer c % 3 without
        // a wait of their own.
        if (lane == 0) {
          int nq = 0, np = 0;
          uint32_t idle = 0;
          uint64_t idle_since = 0;  // time of the first idle poll since the last issue
          while (np < nchunks) {
            bool did = false;
            if (nq < nchunks && nq - 3 < np &&
                (nq < C::kSbuf || mbar_test_wait(bars.sfree(nq % C::kSbuf), ((nq - C::kSbuf) / C::kSbuf) & 1)) &&
                mbar_test_wait(bars.ak(nq & 3), (nq >> 2) & 1)) {
              issue_qk(nq);
              ++nq;
              did = true;
            }
            if (np < nq && mbar_test_wait(bars.pfull(np % 3), (np / 3) & 1) &&
                mbar_test_wait(bars.av(np % 3), (np / 3) & 1)) {
              issue_pv(np);
              ++np;
              did = true;
            }
            if (!did) {
              if (*abort_flag) break;
              ++idle;
              if ((idle & 63) == 0) {
                const uint64_t t = now_ns();
                if (idle_since == 0) {
                  idle_since = t;
                } else if (t - idle_since > kSpinNs || idle >= (1u << 28)) {
                  *abort_flag = 1u;
                  atomicOr(&g_tq_device_error, 1u);
                  break;
                }
              }
            } else {
              idle = 0;
              idle_since = 0;
            }
          }
          // drain before tensor memory is freed
          if (nq > 0) wait_bar(bars.sready((nq - 1) % C::kSbuf), ((nq - 1) / C::kSbuf) & 1, abort_flag, false);
          if (np > 0) wait_bar(bars.pv((np - 1) % 3), ((np - 1) / 3) & 1, abort_flag, false);
        }
      } else if (lane == 0) {
        // ================= MMA issuers (two streams), one thread each, so
        // that the two kinds of MMA are issued in parallel (a batch of eight
        // costs some hundreds of cycles to issue): warp 1 issues S^T(c) once
        // the softmax released S^T buffer c % kSbuf and the keys of chunk c
        // are in tensor memory; warp 0 issues P.V(c) once softmax(c) wrote
        // P'(c) and the values of chunk c are in tensor memory.  P' buffer
        // and value buffer c % 3 are reused for chunk c + 3 only after pv(c),
        // which the softmax and the value dequant wait for.
        int n = 0;
        if (warp == 1) {
          for (int c = 0; c < nchunks; ++c) {
            if (c >= C::kSbuf && !poll_bar(bars.sfree(c % C::kSbuf), ((c - C::kSbuf) / C::kSbuf) & 1, abort_flag))
              break;
            if (!poll_bar(bars.ak(c & 3), (c >> 2) & 1, abort_flag)) break;
            issue_qk(c);
            n = c + 1;
          }
          if (n > 0) wait_bar(bars.sready((n - 1) % C::kSbuf), ((n - 1) / C::kSbuf) & 1, abort_flag, false);
        } else {
          for (int c = 0; c < nchunks; ++c) {
            if (!poll_bar(bars.pfull(c % 3), (c / 3) & 1, abort_flag) ||
                !poll_bar(bars.av(c % 3), (c / 3) & 1, abort_flag))
              break;
            issue_pv(c);
            n = c + 1;
          }
          if (n > 0) wait_bar(bars.pv((n - 1) % 3), ((n - 1) / 3) & 1, abort_flag, false);
        }
      }
      __syncwarp();
    }
  } else if (warp < 8) {
    regs_dec<C::kRegDq>();
    // ================= dequant: thread i = TMEM lane i = token i (keys,
    // parameters) and coordinate i (values)
    const int i = tid - 128;
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    const int pg_i = i >> 4, off_i = i & 15;
    // page p's fields of the chunk in ring stage st at pgf(st, p) + L::kVal / kScale / kZero / kNc
    auto pgf = [&](int st, int p) -> const uint8_t* {
      const uint8_t* stage = sm + C::kRing + st * C::kStageBytes;
      return PRESET == 0 ? stage + C::kRestOff + p * C::kRestBytes - C::kKeyBlock : stage + p * L::kPage;
    };
    // keys and token parameters of chunk c (run one chunk ahead of the values,
    // so that S^T(c + 1) never waits behind P.V(c - 2) freeing A_V)
    auto dq_keys = [&](int c) -> bool {
      const int st = c % C::kStages;
      bool ok = wait_bar(bars.full(st), (c / C::kStages) & 1, abort_flag);
      if (ok && c >= 2)  // A_K[c % 2] read by S^T(c - 2)
        ok = wait_bar(bars.sready((c - 2) % C::kSbuf), ((c - 2) / C::kSbuf) & 1, abort_flag);
      // parameters [c % kColP] were read by softmax(c - kColP) before it
      // released S^T(c - kColP) (two streams), or it ended before softmax(c - 2 -
      // kSbuf) started (64 rows); either release let S^T(c - 2) be issued
      __syncwarp();
      if (!ok) return false;
      const uint8_t* stage = sm + C::kRing + st * C::kStageBytes;
      // keys of token i, all 128 coordinates -> A_K[c % 2]
      const uint32_t ak = tmem + lane_q + C::kTAK + 64 * (c & 1);
      if constexpr (PRESET == 0) {
        // row off_i of page pg_i's key block: 16-byte chunk q sits at q ^ (off_i % 8)
        const uint8_t* kr = stage + pg_i * C::kKeyBlock + off_i * kD;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = *reinterpret_cast<const uint4*>(kr + (((4 * h + q) ^ (off_i & 7)) << 4));
            r[8 * q + 0] = e4m3x2_to_f16x2(w.x);
            r[8 * q + 1] = e4m3x2_to_f16x2(w.x >> 16);
            r[8 * q + 2] = e4m3x2_to_f16x2(w.y);
            r[8 * q + 3] = e4m3x2_to_f16x2(w.y >> 16);
            r[8 * q + 4] = e4m3x2_to_f16x2(w.z);
            r[8 * q + 5] = e4m3x2_to_f16x2(w.z >> 16);
            r[8 * q + 6] = e4m3x2_to_f16x2(w.w);
            r[8 * q + 7] = e4m3x2_to_f16x2(w.w >> 16);
          }
          tmem_st32(ak + 32 * h, r);
        }
      } else {
        // 128 b-bit codes (b = 3, 4, 2): 16 b bytes; pair j (coordinates
        // 2j, 2j+1) at stream bits 2bj .. 2bj + 2b - 1
        constexpr int kB2 = 2 * C::kKeyBits, kW = 4 * C::kKeyBits;  // pair bits, code words
        const uint4* kw =
            reinterpret_cast<const uint4*>(stage + pg_i * L::kPage + L::kKey + off_i * (16 * C::kKeyBits));
        uint32_t wd[kW + 1];
#pragma unroll
        for (int u = 0; u < kW / 4; ++u) {
          const uint4 w = kw[u];
          wd[4 * u + 0] = w.x;
          wd[4 * u + 1] = w.y;
          wd[4 * u + 2] = w.z;
          wd[4 * u + 3] = w.w;
        }
        wd[kW] = 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int bit = kB2 * (32 * h + jj), wi = bit >> 5, sh = bit & 31;
            uint32_t f = wd[wi] >> sh;
            if (sh > 32 - kB2) f |= wd[wi + 1] << (32 - sh);
            r[jj] = pairs[(f & ((1u << kB2) - 1u)) * 32 + lane];
          }
          tmem_st32(ak + 32 * h, r);
        }
      }
      // per-token parameters of token i
      {
        const int pos = (page_lo + c * C::kPages) * kBlock + i;
        const bool valid = pvalid[st * 8 + pg_i] != 0 && pos < t_hi;
        float cs = sl2, sv = 0.f, zv = 0.f;
        int rmin = 1 << 20;
        if (valid) {
          const uint8_t* pg = pgf(st, pg_i);
          if constexpr (PRESET != 0)
            cs = __half2float(*reinterpret_cast<const __half*>(pg + L::kNc + 2 * off_i)) * sl2;
          // odd tokens enter the value operand 16 times larger
          sv = __half2float(*reinterpret_cast<const __half*>(pg + L::kScale + 2 * off_i)) * ((i & 1) ? 0.0625f : 1.f);
          zv = __half2float(*reinterpret_cast<const __half*>(pg + L::kZero + 2 * off_i));
          rmin = 0;
          if (a.causal) {
            const int nmin = pos - L_b + a.n_spec;  // draft n sees this token iff n >= nmin
            rmin = nmin <= 0 ? 0 : max(0, nmin * a.group - row_off);  // first visible row of the tile
          }
        }
        colp[(c % C::kColP) * 128 + i] = make_float4(cs, sv, zv, __int_as_float(rmin));
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars.ak(c & 3));
        mbar_arrive(bars.sready(c % C::kSbuf));
      }
      return true;
    };
    // values of chunk c; then its ring stage is free
    auto dq_values = [&](int c) -> bool {
      const int st = c % C::kStages;
      // A_V[c % 3] was read by P.V(c - 3): done once sready(c) is with one
      // MMA issuer (its commits track every earlier MMA); its own barrier
      // with two
      const bool ok = c < 3 || (C::kStreams == 1 ? wait_bar(bars.sready(c % C::kSbuf), (c / C::kSbuf) & 1, abort_flag)
                                                 : wait_bar(bars.pv(c % 3), ((c - 3) / 3) & 1, abort_flag));
      __syncwarp();
      if (!ok) return false;
      // value codes of coordinate i, all 128 tokens -> A_V[c % 3]: word x of
      // eight codes (token k in bits 4k .. 4k+3) gives the columns
      // (t0, 16 t5) (16 t1, t4) (t2, 16 t7) (16 t3, t6) of its group of 8
      const uint32_t av = tmem + lane_q + C::kTAV + 64 * (c % 3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const uint2 w = *reinterpret_cast<const uint2*>(pgf(st, 4 * h + pp) + L::kVal + 8 * i);
#pragma unroll
          for (int hw = 0; hw < 2; ++hw) {
            const uint32_t x = hw ? w.y : w.x, x8 = x >> 8;
            r[8 * pp + 4 * hw + 0] = x & 0x00F0000Fu;
            r[8 * pp + 4 * hw + 1] = x & 0x000F00F0u;
            r[8 * pp + 4 * hw + 2] = x8 & 0x00F0000Fu;
            r[8 * pp + 4 * hw + 3] = x8 & 0x000F00F0u;
          }
        }
        tmem_st32(av + 32 * h, r);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars.av(c % 3));
        mbar_arrive(bars.empty(st));
      }
      return true;
    };
    bool ok = nchunks == 0 || dq_keys(0);
    for (int c = 0; c < nchunks && ok; ++c) {
      if (c + 1 < nchunks) ok = dq_keys(c + 1);
      ok = ok && dq_values(c);
    }
  } else {
    regs_inc<C::kRegSm>();
    // ================= softmax warpgroup j: thread i = TMEM lane i = token i,
    // query rows [row0, row0 + kRS)
    constexpr int kH = kRS / 2;
    const int j = (warp - 8) >> 2;
    const int sw = warp & 3;
    const int i = sw * 32 + lane;
    const uint32_t lane_q = (uint32_t)(sw * 32) << 16;
    const uint32_t bar_id = 1 + j;
    // 64 rows: rows [32 j, 32 j + 32) of every chunk; two streams: every row
    // of chunks j, j + 2, ...
    constexpr int kStr = C::kStreams;
    const int row0 = kStr == 2 ? 0 : kRS * j;
    const int c0 = kStr == 2 ? j : 0;
    float* red = reinterpret_cast<float*>(sm + C::kRed + j * C::kRedWG);
    float* nms = red;                                      // -m per row
    float* als = red + 32;                                 // rescale factor per row
    float* dlt = red + 64;                                 // m_old - m_new per row (exact path)
    float2* rcs = reinterpret_cast<float2*>(red + 96);     // (2^24 / l, zero term / l)
    float* wmax = red + 160;                               // [4 warps][32 rows] chunk maxima
    float* wsum = red + 288;                               // [2][4 warps][32 rows] l, zero term
    uint32_t* fresh = reinterpret_cast<uint32_t*>(red + 544);  // rows without a maximum yet
    // this token's line of P' (MN-major, swizzled): byte offsets of its 16-byte chunks
    uint32_t poff[kRS / 8];
    {
      const int line = kappa(i);
#pragma unroll
      for (int q = 0; q < kRS / 8; ++q) {
        const uint32_t lg = (uint32_t)((line >> 3) * (8 * C::kLine) + (line & 7) * C::kLine + row0 * 2 + 16 * q);
        poff[q] = lg ^ (((lg >> 7) & ((1u << C::kSwzBits) - 1u)) << 4);
      }
    }
    // m starts at 0 for every row, marked fresh: a row's first visible
    // scores take the exact path, which sets m to their maximum
    if (i < kRS) nms[i] = 0.f;
    if (i == 0) *fresh = kRS == 32 ? 0xFFFFFFFFu : ((1u << kRS) - 1u);
    float2 l2[kH], z2[kH];  // l and the zero term of this token's rows (row pairs)
#pragma unroll
    for (int k = 0; k < kH; ++k) {
      l2[k] = make_float2(0.f, 0.f);
      z2[k] = make_float2(0.f, 0.f);
    }
    named_bar(bar_id, 128);
    const uint32_t s_base = tmem + lane_q + C::kTS + row0;
    bool aborted = false;
    // x: S^T(c) as loaded (one chunk ahead, while the previous chunk's P' is
    // stored), then in place d = s * score_scale - m
    uint32_t x[kRS];
    bool pre = false;  // x already holds (or is loading) S^T(c)
    for (int c = c0; c < nchunks; c += kStr) {
      bool ok = !aborted;
      const bool first = c < kStr;  // this warpgroup's first chunk
      if (!pre) {
        ok = ok && wait_bar(bars.sready(c % C::kSbuf), (c / C::kSbuf) & 1, abort_flag);
        __syncwarp();
        tc_fence_after();
        tmem_ld<kRS>(s_base + NR * (c % C::kSbuf), x);
      }
      tc_wait_ld();
      float4 cp;  // chunk c's parameters for token i (the order is the faster one per mode)
      if constexpr (kStr == 2) cp = colp[(c % C::kColP) * 128 + i];
      // S^T(c) is in registers: its buffer goes back to the MMA issuer (for S^T(c + kSbuf))
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.sfree(c % C::kSbuf));
      if constexpr (kStr == 1) cp = colp[(c % C::kColP) * 128 + i];
      const int rmin = __float_as_int(cp.w);
      const bool masked = __any_sync(kFull, rmin > row0);
      float2* d = reinterpret_cast<float2*>(x);
      // d = s * score_scale - m, masked rows -> -inf
      {
        const float2 cs2 = make_float2(cp.x, cp.x);
        const float4* n4 = reinterpret_cast<const float4*>(nms);
#pragma unroll
        for (int q = 0; q < kRS / 4; ++q) {
          const float4 nv = n4[q];
          d[2 * q] = __ffma2_rn(make_float2(__uint_as_float(x[4 * q]), __uint_as_float(x[4 * q + 1])), cs2,
                                make_float2(nv.x, nv.y));
          d[2 * q + 1] = __ffma2_rn(make_float2(__uint_as_float(x[4 * q + 2]), __uint_as_float(x[4 * q + 3])), cs2,
                                    make_float2(nv.z, nv.w));
        }
        if (masked) {
#pragma unroll
          for (int k = 0; k < kH; ++k) {
            if (row0 + 2 * k < rmin) d[k].x = -CUDART_INF_F;
            if (row0 + 2 * k + 1 < rmin) d[k].y = -CUDART_INF_F;
          }
        }
      }
      float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < kH; k += 2) {
        mx0 = fmax3(mx0, d[k].x, d[k].y);
        if (k + 1 < kH) mx1 = fmax3(mx1, d[k + 1].x, d[k + 1].y);
      }
      // p = 2^d as fp16 pairs (the precision of the P' operand), issued
      // before the vote so that the vote's latency hides behind the
      // exponentials; a vote for the exact path recomputes them.  The first
      // chunk always takes the exact path (every row is fresh), without a
      // vote: each row's largest p is then exactly 1.
      uint32_t ph[kH];
      const uint32_t fr = *fresh;
      bool exact = first;
      if (!first) {
#pragma unroll
        for (int k = 0; k < kH; ++k) ph[k] = ex2_h2(d[k].x, d[k].y);
        // exact path: some score above m + 8 (p could leave the fp16 range),
        // or a row that has no maximum yet sees a score
        bool need = fmaxf(mx0, mx1) > kRescaleThreshold;
        if (fr != 0u) {
#pragma unroll
          for (int k = 0; k < kH; ++k) {
            need |= ((fr >> (2 * k)) & 1u) && d[k].x > -CUDART_INF_F;
            need |= ((fr >> (2 * k + 1)) & 1u) && d[k].y > -CUDART_INF_F;
          }
        }
        // leave the loop together: the named barriers need all four warps
        exact = bar_red_or(bar_id, 128, need || !ok);
      }
      if (exact) {
        if (bar_red_or(bar_id, 128, !ok)) {
          aborted = true;
          break;
        }
        // exact maximum of this chunk for each row over the 128 tokens: a
        // reduce-scatter of d across the warp's lanes (lane l ends with row
        // l % kRS), then across the four warps through shared memory
        {
          float v[kRS];
#pragma unroll
          for (int k = 0; k < kH; ++k) {
            v[2 * k] = d[k].x;
            v[2 * k + 1] = d[k].y;
          }
          warp_transpose_reduce<kRS, true>(v, lane);
          if (lane < kRS) wmax[sw * 32 + lane] = v[0];
        }
        named_bar(bar_id, 128);
        if (i < kRS) {
          const float cm = fmaxf(fmaxf(wmax[i], wmax[32 + i]), fmaxf(wmax[64 + i], wmax[96 + i]));
          float shift = 0.f, al = 1.f;  // m_new = m_old + shift
          if (cm > -CUDART_INF_F) {
            if ((fr >> i) & 1u) {
              shift = cm;  // first visible scores of this row: nothing to rescale
              atomicAnd(fresh, ~(1u << i));
            } else if (cm > 0.f) {
              shift = cm;
              al = ex2(-cm);
            }
          }
          als[i] = al;
          dlt[i] = -shift;
          nms[i] = nms[i] - shift;
        }
        named_bar(bar_id, 128);  // -m and the factors are complete
        bool change = false;
        {
          const float4* a4 = reinterpret_cast<const float4*>(als);
#pragma unroll
          for (int q = 0; q < kRS / 4; ++q) {
            const float4 al4 = a4[q];
            l2[2 * q] = __fmul2_rn(l2[2 * q], make_float2(al4.x, al4.y));
            z2[2 * q] = __fmul2_rn(z2[2 * q], make_float2(al4.x, al4.y));
            l2[2 * q + 1] = __fmul2_rn(l2[2 * q + 1], make_float2(al4.z, al4.w));
            z2[2 * q + 1] = __fmul2_rn(z2[2 * q + 1], make_float2(al4.z, al4.w));
            change |= fminf(fminf(al4.x, al4.y), fminf(al4.z, al4.w)) < 1.0f;
          }
        }
        if (change && !first) {  // uniform across the warpgroup
          // O^T (of this stream) holds its chunks < c: rescale it after the
          // previous one's P.V has landed and before P.V(c) is issued (which
          // needs this warpgroup's pfull); per-stream barriers in two-stream
          // mode, since the other stream may move pv[] on by two phases
          const bool got = kStr == 1 ? wait_bar(bars.pv((c - 1) % 3), ((c - 1) / 3) & 1, abort_flag)
                                     : wait_bar(bars.pvs(j), ((c - 2 - j) >> 1) & 1, abort_flag);
          if (!got) aborted = true;
          __syncwarp();
          tc_fence_after();
#pragma unroll 1
          for (int g = 0; g < kRS / 8; ++g) {
            const uint32_t o_addr = tmem + lane_q + C::kTO + NR * (kStr == 2 ? j : 0) + row0 + 8 * g;
            uint32_t o[8];
            tmem_ld8(o_addr, o);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * als[8 * g + e]);
            tmem_st8(o_addr, o);
          }
          tc_wait_st();
        }
        // d and p again against the new maxima: d + m_old - m_new
        {
          const float4* t4 = reinterpret_cast<const float4*>(dlt);
#pragma unroll
          for (int q = 0; q < kRS / 4; ++q) {
            const float4 tv = t4[q];
            d[2 * q] = __fadd2_rn(d[2 * q], make_float2(tv.x, tv.y));
            d[2 * q + 1] = __fadd2_rn(d[2 * q + 1], make_float2(tv.z, tv.w));
          }
        }
#pragma unroll
        for (int k = 0; k < kH; ++k) ph[k] = ex2_h2(d[k].x, d[k].y);
      }
      // row sums, zero term; P' = p * scale into the MN-major B tile
      uint32_t pk[kH];
      const __half2 svh = __float2half2_rn(cp.y);
      const float2 zv2 = make_float2(cp.z, cp.z);
#pragma unroll
      for (int k = 0; k < kH; ++k) {
        const __half2 ph2 = *reinterpret_cast<const __half2*>(&ph[k]);
        const float2 p = __half22float2(ph2);
        l2[k] = __fadd2_rn(l2[k], p);
        z2[k] = __ffma2_rn(p, zv2, z2[k]);
        const __half2 ps = __hmul2(ph2, svh);
        pk[k] = *reinterpret_cast<const uint32_t*>(&ps);
      }
      // start loading S^T(c + 1) if it is already there (never wait for it here:
      // this chunk's pfull would then depend on S^T(c + 1))
      pre = false;
      if (c + kStr < nchunks) {
        const int cn = c + kStr;
        const bool rdy = mbar_test_wait(bars.sready(cn % C::kSbuf), (cn / C::kSbuf) & 1);
        if (__all_sync(kFull, rdy)) {
          tc_fence_after();
          tmem_ld<kRS>(s_base + NR * (cn % C::kSbuf), x);
          pre = true;
        }
      }
      // P'[c % 3] was read by P.V(c - 3): done since sready(c) is with one MMA
      // issuer; its own barrier with two
      if (C::kStreams == 2 && c >= 3 && !aborted && !wait_bar(bars.pv(c % 3), ((c - 3) / 3) & 1, abort_flag))
        aborted = true;
      uint8_t* pbuf = sm + C::kP + (c % 3) * C::kPBytes;
#pragma unroll
      for (int q = 0; q < kRS / 8; ++q)
        *reinterpret_cast<uint4*>(pbuf + poff[q]) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.pfull(c % 3));
    }
    if (pre) tc_wait_ld();
    // ---- epilogue: l and the zero term of each row over all 128 tokens, by a
    // reduce-scatter across the warp's lanes (each step halves the rows a lane
    // holds) and a sum of the four warps' partials; then the output rows
    // O^T / l straight from tensor memory to global memory
    {
      constexpr int kLanesPerRow = 32 / kRS;
      float v[kRS];
#pragma unroll
      for (int k = 0; k < kH; ++k) {
        v[2 * k] = l2[k].x;
        v[2 * k + 1] = l2[k].y;
      }
      warp_transpose_reduce<kRS, false>(v, lane);
      const float lw = v[0];
#pragma unroll
      for (int k = 0; k < kH; ++k) {
        v[2 * k] = z2[k].x;
        v[2 * k + 1] = z2[k].y;
      }
      warp_transpose_reduce<kRS, false>(v, lane);
      if (lane < kRS) {
        (void)kLanesPerRow;
        wsum[sw * 32 + lane] = lw;
        wsum[128 + sw * 32 + lane] = v[0];
      }
    }
    named_bar(bar_id, 128);
    if constexpr (kStr == 1) {
      if (i < kRS) {
        float lrow = 0.f, zrow = 0.f;
  #pragma unroll
        for (int w = 0; w < 4; ++w) {
          lrow += wsum[w * 32 + i];
          zrow += wsum[128 + w * 32 + i];
        }
        const float inv = lrow > 0.f ? 1.0f / lrow : 0.f;
        rcs[i] = make_float2(inv * 16777216.0f, zrow * inv);  // O^T holds codes as fp16 subnormals (code * 2^-24)
        const int row = row_off + row0 + i;  // row of the kv-head's R
        if (row0 + i < Rt) {
          const float lse = (aborted || *abort_flag) ? CUDART_NAN_F
                                                     : (lrow > 0.f ? (-nms[i] + log2f(lrow)) * kLn2 : -CUDART_INF_F);
          if constexpr (FUSED) {
            a.part_lse[(((long)b * a.Hk + kvh) * a.S + split) * a.R + row] = lse;
          } else {
            const long orow = ((long)(row / a.group) * a.B + b) * a.Hq + kvh * a.group + row % a.group;
            a.part_lse[orow * a.S + split] = lse;
          }
        }
      }
      if (nchunks > 0) {
        const int lc = nchunks - 1;
        if (!aborted && !wait_bar(bars.pv(lc % 3), (lc / 3) & 1, abort_flag)) aborted = true;
        __syncwarp();
        tc_fence_after();
      }
      named_bar(bar_id, 128);  // row constants ready
      aborted = aborted || (*abort_flag != 0u);
      {
        // thread i holds coordinate i of its rows: each row is 32 consecutive
        // floats per warp, one 128-byte store
        uint32_t o[kRS];
        if (nchunks > 0) {
          tmem_ld<kRS>(tmem + lane_q + C::kTO + row0, o);
          tc_wait_ld();
        } else {
  #pragma unroll
          for (int k = 0; k < kRS; ++k) o[k] = 0u;
        }
        if constexpr (FUSED) {
          // the scratch partials of the single-launch verify are laid out
          // [B][Hk][S][R][128] so that a CTA's rows are contiguous
          float* dst = a.part_o + ((((long)b * a.Hk + kvh) * a.S + split) * a.R + row_off + row0) * kD + i;
  #pragma unroll
          for (int k = 0; k < kRS; ++k) {
            const float2 rc = rcs[k];
            if (row0 + k < Rt) dst[k * kD] = aborted ? CUDART_NAN_F : fmaf(__uint_as_float(o[k]), rc.x, rc.y);
          }
        } else {
          int n = (row_off + row0) / a.group, jq = (row_off + row0) % a.group;
  #pragma unroll
          for (int k = 0; k < kRS; ++k) {
            const float2 rc = rcs[k];
            if (row0 + k < Rt) {
              const long orow = ((long)n * a.B + b) * a.Hq + kvh * a.group + jq;
              a.part_o[(orow * a.S + split) * kD + i] = aborted ? CUDART_NAN_F : fmaf(__uint_as_float(o[k]), rc.x, rc.y);
            }
            if (++jq == a.group) {
              jq = 0;
              ++n;
            }
          }
        }
      }
    } else {
      // ---- two streams: stream j publishes (m, l, zero term) of every row;
      // after both streams' last P.V, warpgroup j writes rows
      // [j NR/2, (j + 1) NR/2) as the log-sum-exp merge of the two streams:
      //   out = sum_j a_j (2^24 O_j + z_j) / sum_j a_j l_j,  a_j = 2^(m_j - M)
      constexpr int kHalf = NR / 2;
      float4* stc_mine = reinterpret_cast<float4*>(red + 576);  // [32] (m, l, z, -)
      const float4* stc0 = reinterpret_cast<const float4*>(sm + C::kRed) + 144;
      const float4* stc1 = reinterpret_cast<const float4*>(sm + C::kRed + C::kRedWG) + 144;
      float4* rc4 = reinterpret_cast<float4*>(red + 704);  // [kHalf] (c_0, c_1, zero term, -)
      if (i < kRS) {
        float lrow = 0.f, zrow = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          lrow += wsum[w * 32 + i];
          zrow += wsum[128 + w * 32 + i];
        }
        stc_mine[i] = make_float4(-nms[i], lrow, zrow, 0.f);
      }
      // last chunk of this stream (none if nchunks <= j)
      const int lc = nchunks - 1 >= j ? nchunks - 1 - ((nchunks - 1 - j) & 1) : -1;
      if (lc >= 0) {
        if (!aborted && !wait_bar(bars.pv(lc % 3), (lc / 3) & 1, abort_flag)) aborted = true;
        __syncwarp();
        tc_fence_after();
      }
      named_bar(13, 128 * C::kSW);  // both streams' constants and last P.V
      aborted = aborted || (*abort_flag != 0u);
      const int h0 = j * kHalf;
      if (i < kHalf) {
        const float4 s0 = stc0[h0 + i], s1 = stc1[h0 + i];
        const bool u0 = s0.y > 0.f, u1 = s1.y > 0.f;  // streams that saw the row
        const float M = u0 && u1 ? fmaxf(s0.x, s1.x) : (u0 ? s0.x : s1.x);
        const float a0 = u0 ? ex2(s0.x - M) : 0.f, a1 = u1 ? ex2(s1.x - M) : 0.f;
        const float lsum = a0 * s0.y + a1 * s1.y;
        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
        // O^T holds codes as fp16 subnormals (code * 2^-24)
        rc4[i] = make_float4(a0 * inv * 16777216.0f, a1 * inv * 16777216.0f, (a0 * s0.z + a1 * s1.z) * inv, 0.f);
        const int row = row_off + h0 + i;  // row of the kv-head's R
        if (h0 + i < Rt) {
          const float lse = aborted ? CUDART_NAN_F : (lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -CUDART_INF_F);
          if constexpr (FUSED) {
            a.part_lse[(((long)b * a.Hk + kvh) * a.S + split) * a.R + row] = lse;
          } else {
            const long orow = ((long)(row / a.group) * a.B + b) * a.Hq + kvh * a.group + row % a.group;
            a.part_lse[orow * a.S + split] = lse;
          }
        }
      }
      named_bar(bar_id, 128);
      {
        // thread i holds coordinate i of rows h0 .. h0 + kHalf of both streams
        uint32_t o0[kHalf], o1[kHalf];
#pragma unroll
        for (int k = 0; k < kHalf; ++k) o0[k] = o1[k] = 0u;
        if (nchunks > 0) tmem_ld<kHalf>(tmem + lane_q + C::kTO + h0, o0);
        if (nchunks > 1) tmem_ld<kHalf>(tmem + lane_q + C::kTO + NR + h0, o1);
        tc_wait_ld();
        auto outv = [&](int k) -> float {
          const float4 rc = rc4[k];
          // a stream without visible tokens has weight 0 (its O^T may be unset)
          const float v0 = rc.x != 0.f ? __uint_as_float(o0[k]) * rc.x : 0.f;
          const float v1 = rc.y != 0.f ? __uint_as_float(o1[k]) * rc.y : 0.f;
          return aborted ? CUDART_NAN_F : v0 + v1 + rc.z;
        };
        if constexpr (FUSED) {
          float* dst = a.part_o + ((((long)b * a.Hk + kvh) * a.S + split) * a.R + row_off + h0) * kD + i;
#pragma unroll
          for (int k = 0; k < kHalf; ++k)
            if (h0 + k < Rt) dst[k * kD] = outv(k);
        } else {
          int n = (row_off + h0) / a.group, jq = (row_off + h0) % a.group;
#pragma unroll
          for (int k = 0; k < kHalf; ++k) {
            if (h0 + k < Rt) {
              const long orow = ((long)n * a.B + b) * a.Hq + kvh * a.group + jq;
              a.part_o[(orow * a.S + split) * kD + i] = outv(k);
            }
            if (++jq == a.group) {
              jq = 0;
              ++n;
            }
          }
        }
      }
    }
    if constexpr (FUSED) {
      // ---- stage 2 in the same launch (a cooperative grid: every CTA is
      // resident).  Once all S splits of this (sequence, kv-head) have
      // written their rows, split s merges rows [s rpc, (s + 1) rpc).
      uint32_t* arrived = a.tickets + ((long)b * a.Hk + kvh) * 4;
      uint32_t* merged = arrived + 1;
      volatile uint32_t* go = reinterpret_cast<volatile uint32_t*>(sm + C::kMisc + 8);
      named_bar(15, 128 * C::kSW);  // this CTA's partial rows are written
      if (i == 0 && j == 0) {
        // one release covers the rows every thread of the CTA wrote before the barrier
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(arrived) : "memory");
        *go = spin_until_at_least(arrived, (uint32_t)(a.S * a.rtiles)) ? 1u : 0u;
      }
      named_bar(15, 128 * C::kSW);
      const bool failed = *go == 0u;
      const int nu = a.S * a.rtiles;
      const int rpc = (a.R + nu - 1) / nu, r_lo = unit * rpc, r_hi = min(a.R, r_lo + rpc);
      const int w8 = warp - 8;
      constexpr int kMW = 4 * C::kSW;  // merging warps, a warp per row, lane l: coordinates 4l .. 4l+3
      const long pair_base = ((long)b * a.Hk + kvh) * a.S * a.R;  // split 0, row 0 of this (sequence, kv-head)
      for (int r = r_lo + w8; r < r_hi; r += kMW) {
        const long orow = ((long)(r / a.group) * a.B + b) * a.Hq + kvh * a.group + r % a.group;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f, wl = 0.f;
        for (int t0 = 0; t0 < a.S; t0 += 8) {  // eight partial rows in flight
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = t0 + u < a.S
                       ? __ldcg(reinterpret_cast<const float4*>(a.part_o + (pair_base + (long)(t0 + u) * a.R + r) * kD) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          if (t0 == 0) {
            // weights exp(lse_s - max lse) of all splits (lane s holds split s),
            // loaded while the first rows are in flight
            const float l = lane < a.S ? __ldcg(a.part_lse + pair_base + (long)lane * a.R + r) : -CUDART_INF_F;
            float M = l;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
            wl = (M == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : expf(l - M);
            den = wl;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float w = __shfl_sync(kFull, wl, (t0 + u) & 31);
            if (t0 + u < a.S && w != 0.f) {  // an empty split contributes nothing
              acc.x = fmaf(w, v[u].x, acc.x);
              acc.y = fmaf(w, v[u].y, acc.y);
              acc.z = fmaf(w, v[u].z, acc.z);
              acc.w = fmaf(w, v[u].w, acc.w);
            }
          }
        }
        const float inv = failed ? CUDART_NAN_F : (den > 0.f ? 1.f / den : 0.f);
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        reinterpret_cast<float4*>(a.out + orow * kD)[lane] = acc;
      }
      named_bar(15, 128 * C::kSW);
      if (i == 0 && j == 0 && atomicAdd(merged, 1u) == (uint32_t)(a.S * a.rtiles) - 1u) {
        // every split is past its wait: leave the counters zero for the next call
        atomicExch(arrived, 0u);
        atomicExch(merged, 0u);
        atomicExch(arrived + 2, 0u);
      }
    }
  }

  // ---- teardown: every role has drained its asynchronous work
  tc_fence_before();
  cta_bar();
  if (warp == 1) {
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

template <int PRESET, int NR, bool FUSED>
cudaError_t launch_tc(const VerifyArgs& a, cudaStream_t st) {
  using C = Cfg<PRESET, NR>;
  auto kern = verify_stage1_tc_kernel<PRESET, NR, FUSED>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t bit = 1ull << dev;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.S, a.Hk, a.B * a.rtiles);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  // the single-launch verify waits across CTAs: a cooperative launch
  // guarantees that every CTA of the grid is resident
  attrs[1].id = cudaLaunchAttributeCooperative;
  attrs[1].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = FUSED ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tmap);
}

// how many CTAs of the single-launch verify kernel can be resident at once
template <int PRESET, int NR>
int fused_capacity() {
  using C = Cfg<PRESET, NR>;
  static std::atomic<int> known[64];  // per device: 0 = not queried, else capacity + 1
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = known[dev].load(std::memory_order_acquire);
  if (v == 0) {
    auto kern = verify_stage1_tc_kernel<PRESET, NR, true>;
    int per_sm = 0, sms = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::kThreads, C::kSmem) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      per_sm = sms = 0;
    cudaGetLastError();  // a refused query leaves no sticky error
    v = per_sm * sms + 1;
    known[dev].store(v, std::memory_order_release);
  }
  return v - 1;
}

}  // namespace


// kernel preset of a cache preset: the k3 presets share one kernel
int kernel_preset(int preset) { return preset == 0 || preset == 4 || preset == 5 ? preset : 1; }

template <int P, bool FUSED>
cudaError_t launch_rows(const VerifyArgs& a, cudaStream_t st) {
  if (a.R <= 16) return launch_tc<P, 16, FUSED>(a, st);
  if (a.R <= 32) return launch_tc<P, 32, FUSED>(a, st);
  return launch_tc<P, 64, FUSED>(a, st);
}

template <bool FUSED>
cudaError_t launch_preset(int preset, const VerifyArgs& a, cudaStream_t st) {
  switch (kernel_preset(preset)) {
    case 0: return launch_rows<0, FUSED>(a, st);
    case 4: return launch_rows<4, FUSED>(a, st);
    case 5: return launch_rows<5, FUSED>(a, st);
    default: return launch_rows<1, FUSED>(a, st);
  }
}

template <int P>
int capacity_rows(const VerifyArgs& a) {
  return a.R <= 16 ? fused_capacity<P, 16>() : a.R <= 32 ? fused_capacity<P, 32>() : fused_capacity<P, 64>();
}

cudaError_t launch_verify_stage1_tc(int preset, const VerifyArgs& a, cudaStream_t st) {
  return launch_preset<false>(preset, a, st);
}

bool verify_fused_supported(int preset, const VerifyArgs& a) {
  if (a.S > 32) return false;
  // every CTA resident at once (the merge waits for all splits)
  const long ctas = (long)a.S * a.Hk * a.B * a.rtiles;
  int cap = 0;
  switch (kernel_preset(preset)) {
    case 0: cap = capacity_rows<0>(a); break;
    case 4: cap = capacity_rows<4>(a); break;
    case 5: cap = capacity_rows<5>(a); break;
    default: cap = capacity_rows<1>(a); break;
  }
  return ctas <= cap;
}

cudaError_t launch_verify_fused(int preset, const VerifyArgs& a, cudaStream_t st) {
  return launch_preset<true>(preset, a, st);
}

cudaError_t read_device_error(unsigned int* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tq_device_error, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tq_device_error, &zero, sizeof(unsigned int));
}

}  // namespace tq
