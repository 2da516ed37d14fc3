/*
 * tqkv.h -- C ABI of libtqkv: TurboQuant speculative-verify decode attention
 * over a quantised paged KV cache, hand-written CUDA for sm_103a.
 *
 * The method ("spec-decode-intel-arc", bryanvine.github.io/turboquant-xpu,
 * 2026-04-14):
 *   - section "Context: TurboQuant, speculative decoding, and the gap": keys
 *     are Walsh-Hadamard rotated and coded against a precomputed Lloyd-Max
 *     codebook, values are uniform-scalar quantised with a scale and a zero;
 *     the presets turboquant_k8v4 (FP8 keys, 4-bit values) and
 *     turboquant_k3v4_nc (3-bit keys with norm correction, 4-bit values); the
 *     three hot kernels are the fused store, decode stage 1 and the stage 2
 *     reduction;
 *   - section "Roofline": the cache is blocks x 16 tokens x Hk x slot, the
 *     k8v4 slot is 196 bytes;
 *   - section "Part 3: The fused Triton kernel": all N_spec draft queries of a
 *     sequence are processed in one launch and share one K dequant per tile;
 *   - section "Part 4: The causal correction": draft query n attends to
 *     cached_len + n + 1 tokens;
 *   and "sycl-three-attempts-arc-b70" (2026-04-15), section "Part 3:
 *   joint_matrix + split-KV": NUM_KV_SPLITS partial attention per (b, h_q),
 *   then a log-sum-exp reduction over the splits.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers into caller-owned memory; the
 *     library never allocates, frees or keeps per-call state, and only
 *     tq_device_status and the set-up of tq_verify_noalloc synchronise (the
 *     sticky error word and tq_verify_noalloc's scratch are the library's
 *     only device state).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     only enqueued; results are ready when the stream reaches that point.
 *   - Arguments are validated on the host before anything is launched.  On
 *     error nothing is enqueued and a tq_status other than TQ_OK is returned;
 *     no entry point aborts, throws or prints.
 *   - Element types: fp16 = IEEE binary16, fp32 = IEEE binary32, all arrays
 *     dense row-major (C order) in the index order written below.
 *   - Head dimension D is 128 and the cache block (page) holds 16 tokens.
 */
#ifndef TQKV_H
#define TQKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size   */
  TQ_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement  */
  TQ_ERR_MISALIGNED = 3,  /* a pointer lacks the alignment stated below    */
  TQ_ERR_CUDA = 4,        /* the CUDA runtime reported a launch error      */
  TQ_ERR_TIMEOUT = 5      /* a bounded device-side wait expired            */
} tq_status;

typedef enum {
  TQ_PRESET_K8V4 = 0,     /* keys e4m3 (RNE, saturating), values 4-bit         */
  TQ_PRESET_K3V4_NC = 1,  /* keys: WHT + 3-bit Lloyd-Max codes + fp16 norm
                             correction |k| / |c_hat|; values 4-bit            */
  TQ_PRESET_K3V4 = 2,     /* as k3v4_nc (same page), but the fp16 key factor is
                             the plain norm |k| (no correction)                */
  TQ_PRESET_K3V4_NC_RS = 3, /* as k3v4_nc, keys rotated by H diag(s) / sqrt(128):
                             s_j = -1 where the top bit of output j of
                             SplitMix64 seeded 0x54515F5349474E53 is set      */
  TQ_PRESET_K4V4_NC = 4,  /* as k3v4_nc with 4-bit codes of the 16-level
                             Lloyd-Max codebook (the "3-4 bit" widths of the
                             "Context" section)                                */
  TQ_PRESET_K2V4_NC = 5   /* as k3v4_nc with 2-bit codes of the 4-level
                             Lloyd-Max codebook                                */
} tq_preset;

/* Description of a caller-owned paged cache in device memory.
 * Layout: u8 [num_blocks][num_kv_heads][tq_page_bytes(preset)].  One page is
 * the 16 tokens of one block for one kv-head, stored planar:
 *   k8v4    (3136 B = 16 x 196): K e4m3 [16][128] @0 | V codes [128][8] @2048
 *           | V scale fp16 [16] @3072 | V zero fp16 [16] @3104
 *   k3v4_nc (1920 B = 16 x 120): K codes [16][48] @0 | K nc fp16 [16] @768
 *           | V codes [128][8] @800 | V scale fp16 [16] @1824
 *           | V zero fp16 [16] @1856 | 32 B padding @1888 (never written)
 *   k4v4_nc (2176 B = 16 x 136): K codes [16][64] @0 | K nc fp16 [16] @1024
 *           | V codes [128][8] @1056 | V scale @2080 | V zero @2112
 *           | 32 B padding @2144
 *   k2v4_nc (1664 B = 16 x 104): K codes [16][32] @0 | K nc fp16 [16] @512
 *           | V codes [128][8] @544 | V scale @1568 | V zero @1600
 *           | 32 B padding @1632
 * (k3v4 and k3v4_nc_rs use the k3v4_nc page.)  V codes are coordinate-major:
 * byte 8d + t/2 holds the 4-bit code of coordinate d for token t of the page
 * (low nibble for even t).  The b-bit key codes of a token (b = 3, 4, 2) form
 * a little-endian bit stream, code j at bits bj..bj+b-1.
 * `cache` must be 16-byte aligned. */
typedef struct {
  int32_t preset;       /* tq_preset                                  */
  int32_t head_dim;     /* must be 128                                */
  int32_t block_size;   /* must be 16                                 */
  int32_t num_kv_heads; /* Hk >= 1                                    */
  int32_t num_blocks;   /* >= 0                                       */
  int32_t reserved;     /* must be 0                                  */
  void* cache;          /* device pointer, see layout above           */
} tq_cache_desc;

/* Bytes of one (block, kv-head) page: 3136 (k8v4), 1920 (k3 presets), 2176
 * (k4v4_nc), 1664 (k2v4_nc), 0 for an unknown preset.  16 x the slot size of
 * the "Roofline" section (196 B for k8v4; 120 B for k3v4_nc; the other widths
 * rounded up to 4 bytes the same way). */
size_t tq_page_bytes(int32_t preset);

/* Levels of a preset's key codebook: 8 (k3 presets), 16 (k4v4_nc), 4
 * (k2v4_nc), 0 for k8v4 or an unknown preset. */
int32_t tq_key_levels(int32_t preset);

/* Bytes of the stage-1 partials for one call: partial_o (fp32
 * [n_spec][B][Hq][num_kv_splits][128]) plus partial_lse (fp32
 * [n_spec][B][Hq][num_kv_splits]).  0 if an argument is < 1. */
size_t tq_partials_bytes(int32_t n_spec, int32_t B, int32_t Hq, int32_t num_kv_splits);

/* A preset's key codebook: the n-level Lloyd-Max quantiser of N(0, 1/128),
 * n = tq_key_levels(preset) ("Context" section: a precomputed Lloyd-Max
 * codebook), derived in fp64 at first use and rounded to fp16; written
 * ascending to the HOST array centroids_out[n] as the fp32 values of those
 * fp16 numbers.  Returns TQ_ERR_UNSUPPORTED for k8v4 (no codebook),
 * TQ_ERR_INVALID_ARG for NULL or an unknown preset. */
tq_status tq_codebook(int32_t preset, float* centroids_out);

/* Static English text for a status code (never NULL). */
const char* tq_status_string(int32_t status);

/* Fused store ("Context" section: the fused store kernel): quantise and pack
 * T new tokens into the cache.
 *   k, v          fp16 [T][num_kv_heads][128], 16-byte aligned
 *   slot_mapping  int32 [T], 4-byte aligned: slot = block * 16 + offset;
 *                 a negative slot or one >= num_blocks * 16 skips that token
 * Per token-head, k8v4 writes the e4m3 key bytes; k3v4_nc computes |k|, the
 * rotation H k, the nearest centroid of each coordinate of H k / (|k| sqrt 128)
 * and nc = |k| / |c_hat| (fp16).  Values (both presets): zero = min, scale =
 * (max - min) / 15 rounded up to fp16, codes = rint((v - zero) / scale)
 * clamped to [0, 15].  The bytes are a deterministic function of k and v
 * (fixed fp32 operation order).  T == 0 enqueues nothing.  Two tokens mapped
 * to the same slot race (the last write of either wins per byte). */
tq_status tq_store(const tq_cache_desc* cache, const void* k, const void* v,
                   const int32_t* slot_mapping, int32_t T, void* stream);

/* Spec-verify stage 1 ("Part 3" / "Part 4" sections and split-KV of
 * "sycl-three-attempts"): partial softmax attention of every draft query over
 * one of num_kv_splits ranges of its sequence's cached tokens.
 *   q             fp16 [n_spec][B][Hq][128], 16-byte aligned
 *   block_table   int32 [B][max_blocks], 4-byte aligned: the cache block of
 *                 each 16-token page of each sequence; an id outside
 *                 [0, num_blocks) makes that page's tokens invisible
 *   seq_lens      int32 [B], 4-byte aligned: tokens of each sequence in the
 *                 cache, INCLUDING its n_spec draft tokens (clamped to
 *                 [0, max_blocks * 16])
 *   causal        1: draft n of sequence b sees positions < L_b - n_spec + n + 1
 *                 (cached_len + n + 1 with cached_len = L_b - n_spec);
 *                 0: every draft sees all L_b positions (parallel completion)
 *   partial_o     fp32 [n_spec][B][Hq][num_kv_splits][128], 16-byte aligned
 *   partial_lse   fp32 [n_spec][B][Hq][num_kv_splits], 4-byte aligned
 * Query head h uses kv-head h / (Hq / num_kv_heads) (GQA).  Split s covers
 * positions [s * c, (s + 1) * c) with c = 16 * ceil(ceil(L_b / S) / 16).  For
 * each (n, b, h, s): partial_o = softmax-weighted mean of the decoded values
 * over the visible positions of the split, partial_lse = ln(sum exp(score))
 * with score = q . k_hat / sqrt(128); an empty range gives partial_o = 0 and
 * partial_lse = -inf.  Requires 1 <= n_spec <= 128, Hq % num_kv_heads == 0,
 * R = n_spec * Hq / num_kv_heads <= 1024 (the rows of one kv-head: up to 16
 * drafts at GQA 8, or a continuation chunk of up to 128 query tokens; rows
 * beyond 64 are tiled 64 per CTA over the same pages), 1 <= num_kv_splits <=
 * 65535, B * ceil(R / 64) <= 65535; otherwise TQ_ERR_UNSUPPORTED. */
tq_status tq_verify_stage1(const tq_cache_desc* cache, const void* q, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* seq_lens, int32_t n_spec, int32_t B,
                           int32_t Hq, int32_t num_kv_splits, int32_t causal, float* partial_o,
                           float* partial_lse, void* stream);

/* Spec-verify stage 2 ("Roofline" section: the stage-2 reduction kernel):
 * log-sum-exp merge of the splits,
 *   out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M),  M = max_s lse_s,
 * and out = 0 for a row whose splits are all empty.
 *   partial_o, partial_lse  as written by tq_verify_stage1 (same alignment)
 *   out                     fp32 [n_spec][B][Hq][128], 16-byte aligned
 * head_dim must be 128. */
tq_status tq_verify_stage2(const float* partial_o, const float* partial_lse, int32_t n_spec,
                           int32_t B, int32_t Hq, int32_t head_dim, int32_t num_kv_splits,
                           float* out, void* stream);

/* Both stages of one verify call: the attention output of every draft x
 * query head, as tq_verify_stage1 followed by tq_verify_stage2 (the
 * split-KV partial attention, "sycl-three-attempts-arc-b70" section "Part 3",
 * and its log-sum-exp merge).  The pages run the two stages as two launches.
 * Here, when num_kv_splits <= 32 and all num_kv_splits * Hk * B *
 * ceil(R / 64) CTAs fit on the device at once, one cooperative launch runs
 * both: every CTA (split s, row tile t of its (sequence, kv-head) pair;
 * unit u = t S + s) writes its partial rows, counts itself in on the pair's
 * arrival counter, waits (bounded) until all S ceil(R / 64) CTAs of the pair
 * have, then merges its share of the rows (rows [u r, (u + 1) r),
 * r = ceil(R / (S ceil(R / 64)))).  Otherwise stage 1 and stage 2 are
 * enqueued as two launches.
 * Arguments, layouts, alignment and validation are those of
 * tq_verify_stage1 (its first twelve arguments; the partials are scratch
 * here and their contents unspecified afterwards) plus
 *   tickets  u32 [B][Hk][4], 4-byte aligned, caller-owned: must be all zero
 *            before the first call and is all zero again after each call
 *            completes (entries 0, 1 and 2 of each pair are its arrival,
 *            completion and stored-draft counters, entry 3 is unused); calls
 *            that share a tickets buffer must not overlap in time (order them
 *            on one stream);
 *   out      fp32 [n_spec][B][Hq][128], 16-byte aligned; written.
 * A cross-split wait that expires writes NaN rows and sets the device error
 * word (tq_device_status); the counters may then be left non-zero, so after
 * a call that set the error word the caller zeroes tickets again before the
 * next call. */
tq_status tq_verify(const tq_cache_desc* cache, const void* q, const int32_t* block_table,
                    int32_t max_blocks, const int32_t* seq_lens, int32_t n_spec, int32_t B,
                    int32_t Hq, int32_t num_kv_splits, int32_t causal, float* partial_o,
                    float* partial_lse, uint32_t* tickets, float* out, void* stream);

/* One verify step: store each sequence's n_spec draft tokens into the cache
 * (tq_store), then verify them (tq_verify).  The pages run the store and the
 * attention as separate kernels ("spec-decode-intel-arc", section "Context":
 * the fused store is one of the three hot kernels; section "Part 3").  Draft n
 * of sequence b goes to position p = min(seq_lens[b], max_blocks * 16) -
 * n_spec + n, i.e. page block_table[b][p / 16], offset p % 16 (a negative p
 * or an out-of-range block id skips the draft), with the bytes tq_store
 * writes.  Where tq_verify runs as one launch, the drafts are stored inside
 * it: CTA unit u of the pair stores drafts n = u mod (S ceil(R / 64)) while
 * its first pages are in flight and counts them on the pair's draft counter
 * (tickets entry 2); a CTA whose page range holds drafts copies those pages
 * only after all n_spec are counted (bounded wait).  Otherwise a store launch
 * and tq_verify are enqueued.
 * Arguments are those of tq_verify plus
 *   k_new, v_new  fp16 [B][n_spec][Hk][128], 16-byte aligned: the drafts'
 *                 keys and values (the cache is written, so it must not be
 *                 read by other work in flight). */
tq_status tq_store_verify(const tq_cache_desc* cache, const void* k_new, const void* v_new, const void* q,
                          const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                          int32_t n_spec, int32_t B, int32_t Hq, int32_t num_kv_splits, int32_t causal,
                          float* partial_o, float* partial_lse, uint32_t* tickets, float* out, void* stream);

/* tq_verify without caller scratch (paper has no counterpart: a convenience
 * of this C ABI).  The partials, log-sum-exps and merge counters live in
 * device arrays of the library itself (16 MiB of partials and log-sum-exps,
 * 16384 counter words), so a call allocates nothing; out is the only buffer
 * written.  Arguments, layouts, alignment and validation are those of
 * tq_verify without partial_o, partial_lse and tickets.
 *   Set-up: the first call on a device looks up the arrays' addresses and
 *     clears the counters, synchronising the device; make it before any
 *     stream capture on that device.  After tq_device_status has reported an
 *     expired wait, the next call on every device sets the scratch up again
 *     (the counters may have been left non-zero), so that call too must come
 *     before any capture.
 *   Sharing: every call on a device uses the same scratch.  Calls on one
 *     device must not overlap in time (order them on one stream); calls that
 *     run concurrently on different streams race on the scratch.
 *   Errors: TQ_ERR_UNSUPPORTED when n_spec * B * Hq * num_kv_splits * 129
 *     floats exceed the scratch or B * Hk * 4 exceeds the counter words (the
 *     caller then uses tq_verify with its own buffers); TQ_ERR_CUDA when the
 *     set-up fails; otherwise tq_verify's status. */
tq_status tq_verify_noalloc(const tq_cache_desc* cache, const void* q, const int32_t* block_table,
                            int32_t max_blocks, const int32_t* seq_lens, int32_t n_spec, int32_t B,
                            int32_t Hq, int32_t num_kv_splits, int32_t causal, float* out, void* stream);

/* Reads and clears the library's sticky device-side error word on the
 * current device.  Every wait of the tensor-core stage-1 kernel on a shared
 * memory barrier is bounded; when one expires the kernel gives up on its
 * (split, kv-head, sequence), writes NaN partials for it and sets the word.
 * Returns TQ_ERR_TIMEOUT if that happened since the last call, TQ_OK if not,
 * TQ_ERR_CUDA if the word could not be read.  Synchronises the device (it is
 * a diagnostic, not a per-call step). */
tq_status tq_device_status(void);

#ifdef __cplusplus
}
#endif

#endif /* TQKV_H */
