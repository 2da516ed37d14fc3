// tq_common.cuh -- page layout, launch parameters and small device helpers
// shared by the store and verify kernels of libtqkv (internal header).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tq {

constexpr int kD = 128;      // head dimension
constexpr int kBlock = 16;   // tokens per cache block (page)

// Planar page of one (block, kv-head): the byte budgets of the two presets
// (k8v4 slot 196 B as in the "Roofline" section of spec-decode-intel-arc;
// k3v4_nc slot 118 B aligned to 120 B).
struct K8 {
  static constexpr int kKey = 0;      // e4m3 [16][128]
  static constexpr int kVal = 2048;   // codes [128 coord][8 B: 16 tokens]
  static constexpr int kScale = 3072; // fp16 [16]
  static constexpr int kZero = 3104;  // fp16 [16]
  static constexpr int kPage = 3136;
};
struct K3 {
  static constexpr int kKey = 0;      // 3-bit codes [16][48]
  static constexpr int kNc = 768;     // fp16 [16]
  static constexpr int kVal = 800;    // codes [128 coord][8 B: 16 tokens]
  static constexpr int kScale = 1824; // fp16 [16]
  static constexpr int kZero = 1856;  // fp16 [16]
  static constexpr int kPage = 1920;  // 32 B padding at 1888
};

// the other key widths: 4-bit (16-level) and 2-bit (4-level) codes, the
// k3v4_nc page with slots of 134 B and 102 B rounded up to 4 bytes
struct K4 {
  static constexpr int kKey = 0;      // 4-bit codes [16][64]
  static constexpr int kNc = 1024;    // fp16 [16]
  static constexpr int kVal = 1056;   // codes [128 coord][8 B: 16 tokens]
  static constexpr int kScale = 2080; // fp16 [16]
  static constexpr int kZero = 2112;  // fp16 [16]
  static constexpr int kPage = 2176;  // 32 B padding at 2144
};
struct K2 {
  static constexpr int kKey = 0;      // 2-bit codes [16][32]
  static constexpr int kNc = 512;     // fp16 [16]
  static constexpr int kVal = 544;    // codes [128 coord][8 B: 16 tokens]
  static constexpr int kScale = 1568; // fp16 [16]
  static constexpr int kZero = 1600;  // fp16 [16]
  static constexpr int kPage = 1664;  // 32 B padding at 1632
};

// Kernel presets: 0 = k8v4, 1 = the k3 presets (k3v4_nc, k3v4, k3v4_nc_rs
// differ in runtime flags only), 4 = k4v4_nc, 5 = k2v4_nc.
template <int PRESET>
struct Layout;
template <>
struct Layout<0> : K8 {};
template <>
struct Layout<1> : K3 {};
// k3v4: k3v4_nc's page, the plain norm |k| as key factor
template <>
struct Layout<2> : K3 {};
template <>
struct Layout<4> : K4 {};
template <>
struct Layout<5> : K2 {};

// bits per key code (0: FP8 keys)
template <int PRESET>
__host__ __device__ constexpr int key_bits() {
  return PRESET == 0 ? 0 : PRESET == 4 ? 4 : PRESET == 5 ? 2 : 3;
}

// Up to sixteen fp16 centroids, ascending (8 for the k3 presets, 16 for
// k4v4_nc, 4 for k2v4_nc), passed to kernels by value.
struct Codebook {
  uint16_t c[16];
};

struct StoreArgs {
  uint8_t* cache;
  int num_blocks;
  int Hk;
  const __half* k;
  const __half* v;
  const int32_t* slots;  // [T]; null: the drafts of a verify step, slots from the block table
  int T;
  // with slots == null: token t = b * n_spec + n goes to position
  // min(seq_lens[b], max_blocks * 16) - n_spec + n of sequence b
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  int n_spec;
  int plain_norm;      // preset k3v4: the plain norm as key factor
  uint32_t signs[4];   // preset k3v4_nc_rs: bit j set where coordinate j's sign is flipped
  Codebook cb;
};

struct VerifyArgs {
  const uint8_t* cache;
  int num_blocks;
  int Hk;
  const __half* q;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  int n_spec, B, Hq, group, R, S, causal;
  int rtiles;         // row tiles of up to 64 rows per (split, kv-head, sequence): ceil(R / 64)
  float* part_o;
  float* part_lse;
  float* out;         // merged output (single-launch verify only)
  uint32_t* tickets;  // [B][Hk][4], zero between calls (single-launch verify only)
  // drafts to store first (single-launch store + verify only, else null):
  // fp16 [B][n_spec][Hk][128], draft n of sequence b at position L_b - n_spec + n
  const __half* dk;
  const __half* dv;
  uint8_t* cache_w;   // the cache, writable (same as cache)
  int plain_norm;     // preset k3v4: drafts stored with the plain norm as key factor
  uint32_t signs[4];  // preset k3v4_nc_rs: bit j set where coordinate j's sign is flipped
  Codebook cb;
};

struct MergeArgs {
  const float* part_o;
  const float* part_lse;
  float* out;
  long rows;
  int S;
};

// Programmatic dependent launch.  Every kernel of the library waits for the
// previous grid in its stream (and the visibility of its writes) before it
// touches global memory, and at once allows the next grid to be scheduled, so
// that launch processing and block dispatch overlap the previous kernel.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Host-side launchers (each returns the cudaError_t of its launch).
cudaError_t launch_store(int preset, const StoreArgs& a, cudaStream_t st);
cudaError_t launch_verify_stage1(int preset, const VerifyArgs& a, cudaStream_t st);
cudaError_t launch_verify_stage2(const MergeArgs& a, cudaStream_t st);
// stage 1 on the tensor cores (tcgen05); rows beyond 64 per kv-head are
// tiled across CTAs
cudaError_t launch_verify_stage1_tc(int preset, const VerifyArgs& a, cudaStream_t st);
// both stages in one cooperative launch (S <= 32, every CTA resident at once)
bool verify_fused_supported(int preset, const VerifyArgs& a);
cudaError_t launch_verify_fused(int preset, const VerifyArgs& a, cudaStream_t st);
// sticky device-side error word (nonzero after a bounded wait expired)
cudaError_t read_device_error(unsigned int* out, bool clear);
// after an expired wait the merge counters of tq_verify_noalloc's scratch may
// be left non-zero: its next call on every device sets the scratch up again
void noalloc_mark_stale();

}  // namespace tq
