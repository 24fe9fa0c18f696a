/*
 * kvq.h - C ABI of the rotated low-bit KV-cache library (libkvq.so).
 *
 * Two cache formats, each with a quantise-on-append call and a fused
 * packed-cache decode-attention call, plus two host-only helpers:
 *
 *   INT2     "Output-Aware Rotation for INT2 KV-Cache Quantization":
 *            keys centred per head (§1, attention-equivalent
 *            reparameterisation), rotated z = (k - mu) R_k and values
 *            w = v R_v (§3.1 Eq. 4, row-vector convention), then INT2 group
 *            quantisation Q2 with groups of 32 rotated channels and fp16
 *            (scale, min) per group (§1: all values of a group share one
 *            scale; clip ratio c = 1).  Decode attends in the rotated basis
 *            (§3 Eqs. 1-2 with Eq. 4 folded in): q' = q R_k once per query
 *            head, o' = sum_s p_s Q2(w_s), o = o' R_v^T once.
 *   Block-GTQ "RoPE-Aware Bit Allocation for KV-Cache Quantization":
 *            greedy per-RoPE-block widths (prerequisites, Theorem 1; method
 *            step 2), grouped TQ-MSE key encoding (step 3), uniform TQ-MSE
 *            values (step 4), packed-cache decode (Figure 2).
 *
 * Conventions (all calls):
 *  - d (head dimension) must be 128; the page size is 16 tokens.
 *  - Device pointers are owned by the caller; the library allocates no
 *    memory at call time.  Its global state: the thread-local error text,
 *    per-device caches (SM count, kernel shared-memory opt-ins), the fixed
 *    scratch array of kvq_decode_attn_int2_noalloc and the one-shot flag of
 *    the test hook kvq_debug_drop_next_copy.
 *  - Device work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and is asynchronous: faults surface at the caller's
 *    next synchronisation.  Argument errors are detected on the host before
 *    any launch and returned as a kvq_status; nothing is launched then.
 *  - Tensors are dense row-major: k, v [n_tok][H_kv][d] bf16;
 *    q [B][H_q][d] bf16; out [B][H_q][d] fp32; block_table [B][max_pages]
 *    int32 physical page ids; context_lens [B] int32 tokens to attend.
 *  - Query head j reads KV head j / (H_q / H_kv) (contiguous GQA groups).
 *  - slot_mapping[t] = page * 16 + slot; -1 skips token t.
 *  - Kernels are launched with programmatic dependent launch: a call's
 *    kernel may start while the kernel before it in the stream is still
 *    running, and waits for it before reading any input (before the wait it
 *    only asks L2 to prefetch lines, which returns no data), so every input,
 *    rotations included, may be written by the kernel just before the call.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = -1,     /* bad size, null pointer, misalignment */
    KVQ_ERR_UNSUPPORTED = -2,     /* d != 128, GQA group > 8, widths > 8 ... */
    KVQ_ERR_WORKSPACE = -3,       /* workspace too small */
    KVQ_ERR_CUDA = -4,            /* a CUDA runtime call failed */
    KVQ_ERR_BAD_BLOCK_TABLE = -5  /* reported by kvq_workspace_status */
} kvq_status;

/* Text of the last error on this thread ("" if none). */
const char* kvq_last_error(void);

/* ------------------------------------------------------------------ INT2 */

/* Bytes of one (page, KV head) tile of the INT2 cache (1536 at d = 128):
 *   [   0,  512) K codes, 16 slots x 32 B
 *   [ 512,  768) K meta, 16 slots x 4 groups x (fp16 scale, fp16 min)
 *   [ 768, 1280) V codes
 *   [1280, 1408) V scales, 8 slot pairs x 4 groups x (fp16 of slot 2j, of slot 2j+1)
 *   [1408, 1536) V mins, the same layout
 * The cache is tiles[num_pages][H_kv].  A 32-byte code record stores
 * channel 32*g + 4*b + c (g = 0..3 group, b = 0..7, c = 0..3) in bits
 * 2c..2c+1 of byte 4*b + g.  The value scale of slot s, group g is at byte
 * 1280 + 16*(s/2) + 4*g + 2*(s%2), its min 128 bytes later.  Returns 0 for
 * unsupported d. */
size_t kvq_int2_tile_bytes(int d);

/* Quantise-on-append of n_tok tokens into the INT2 cache.
 *   k, v      device bf16 [n_tok][H_kv][d]
 *   mu_k      device fp32 [H_kv][d] key centre (fixed offline)
 *   R_k, R_v  device fp32 [H_kv][d][d] orthogonal rotations, row-major,
 *             applied as z = (k - mu_k) R_k, w = v R_v
 *   cache     device, num_pages * H_kv * kvq_int2_tile_bytes(d) bytes
 *   dbg_rot_k, dbg_rot_v  nullable device fp32 [n_tok][H_kv][d]: the
 *             rotated vectors the codes were decided from
 *   err_count nullable device int32: incremented once per token whose
 *             slot lies outside [0, num_pages*16) (other than -1); such
 *             tokens are skipped.
 * Each rotated coordinate is an fp32 fused-multiply-add chain over the
 * input coordinates in ascending order; per 32-channel group
 * scale = fp16(fp32(fp32(max - min) / 3)), min = fp16(min) (saturating at
 * +-65504); code = number of thresholds min + (c + 1/2) scale (c = 0..2)
 * strictly below the value (ties to the lower level), 0 when scale == 0.
 * Tokens with equal slots race (last writer unspecified).  Appends of 256
 * tokens or more with 16-byte aligned k, v (and exports) take a
 * register-tiled kernel (R in shared memory, about 100 KB per CTA, opted in on
 * first use); it runs the same chains, so the cache bytes and exports are
 * identical to those of smaller calls. */
kvq_status kvq_append_int2(const void* k, const void* v, int n_tok, int H_kv, int d,
                           const int32_t* slot_mapping, const float* mu_k,
                           const float* R_k, const float* R_v,
                           void* cache, int64_t num_pages,
                           float* dbg_rot_k, float* dbg_rot_v, int32_t* err_count,
                           void* stream);

/* kvq_append_int2 with clip ratio c of Q2(.; c, G) ("Output-Aware Rotation
 * for INT2 KV-Cache Quantization" §3.1, Eq. (4) names c without a value):
 * each group's range ends scale to c*min and c*max (fp32 products), so
 * values beyond the clipped range saturate at codes 0 and 3.  0 < clip <= 1;
 * clip = 1 is kvq_append_int2 exactly.  Other arguments as kvq_append_int2. */
kvq_status kvq_append_int2_clip(const void* k, const void* v, int n_tok, int H_kv, int d,
                                const int32_t* slot_mapping, const float* mu_k,
                                const float* R_k, const float* R_v, float clip,
                                void* cache, int64_t num_pages,
                                float* dbg_rot_k, float* dbg_rot_v, int32_t* err_count,
                                void* stream);

/* Reads cached tokens back: the dequantised rotated key and value vectors
 * of the tokens at slot_mapping[0..n), each coordinate min + code * scale as
 * one fp32 fused multiply-add (the Q2(zR) of Eq. (4), still in the rotated
 * basis: multiply by R^T, and add mu for keys, for the original basis).
 *   cache         as written by the append calls (num_pages pages)
 *   slot_mapping  device int32 [n]; a slot outside the cache gives zeros
 *   k_rot, v_rot  device fp32 [n][H_kv][d], either may be null
 * Enqueued on `stream`. */
kvq_status kvq_dequant_int2(const void* cache, int64_t num_pages, int H_kv, int d,
                            const int32_t* slot_mapping, int n, float* k_rot, float* v_rot,
                            void* stream);

/* Bytes of decode workspace for B sequences, H_q query heads, H_kv KV heads
 * and num_splits split-K partitions per (sequence, KV head), enough for every
 * decode entry point called with that num_splits (num_splits = 0: room for
 * the automatic choice of each, kvq_decode_attn_int2, its BF16-window form
 * and bgtq_decode_attn, at max_pages_per_seq pages on the current device,
 * whose SM count sets the automatic choice).  The workspace holds an error
 * word, a split ticket per (sequence, KV head) and the split partials.  It
 * must be zero-filled once before its first use; every call leaves its
 * tickets at zero again.  Returns 0 for invalid sizes (max_pages_per_seq
 * above 2^28 among them). */
size_t kvq_decode_workspace_bytes(int B, int H_q, int H_kv, int max_pages_per_seq, int num_splits);

/* The split count per (sequence, KV head) the automatic choice (num_splits =
 * 0) of bgtq_decode_attn uses: the most splits that keep B * H_kv * splits
 * within one wave of one CTA per SM of the current device (152 on a GB300,
 * and where no device can be queried), at least 1, at most one split per 32
 * pages and at most 256.  (The INT2 decode's automatic choice is described
 * at kvq_decode_attn_int2.) */
int kvq_decode_auto_splits(int B, int H_q, int H_kv, int max_pages_per_seq);

/* Fused packed-cache decode attention over the INT2 cache.
 *   q            device bf16 [B][H_q][d]
 *   cache        as written by kvq_append_int2 (num_pages pages)
 *   block_table  device int32 [B][max_pages_per_seq]
 *   context_lens device int32 [B], 0 <= len <= 16 * max_pages_per_seq
 *   R_k, R_v     as for append
 *   scale        logit scale (1/sqrt(d) for Eq. 1)
 *   out          device fp32 [B][H_q][d]: o = softmax(q'.Q2(z)*scale) Q2(w) R_v^T
 *                (zeros for an empty context)
 *   workspace    device, >= kvq_decode_workspace_bytes(...), zeroed once
 *   num_splits   CTAs per (sequence, KV head), at most 254: the B * H_kv
 *                units are laid end to end as B * H_kv * max_pages_per_seq
 *                pages and num_splits * B * H_kv CTAs take equal shares of
 *                them; 0 = automatic: one CTA per SM of the device (at least
 *                one per unit, at most one per 32 pages)
 * Each CTA publishes an unrotated split partial per unit its share covers;
 * the last to finish merges them and applies R_v^T once.  Block-table
 * entries outside [0, num_pages) are not read: their tokens are dropped and
 * kvq_workspace_status reports KVQ_ERR_BAD_BLOCK_TABLE. */
kvq_status kvq_decode_attn_int2(const void* q, int B, int H_q, int H_kv, int d,
                                const void* cache, int64_t num_pages,
                                const int32_t* block_table, int max_pages_per_seq,
                                const int32_t* context_lens,
                                const float* R_k, const float* R_v, float scale,
                                float* out, void* workspace, size_t workspace_bytes,
                                int num_splits, void* stream);

/* One decode step of one layer in a single launch: kvq_append_int2 of the
 * new token followed by kvq_decode_attn_int2 ("Output-Aware Rotation for
 * INT2 KV-Cache Quantization" §1 and §3.1 Eq. 4 for the append, §3 Eqs. 1-2
 * for the attention).  For every sequence b with ctx = context_lens[b] >= 1
 * the new token k_new[b], v_new[b] ([B][H_kv][d] bf16, original basis, key
 * not centred) is quantised exactly as kvq_append_int2 does it and written
 * to position ctx - 1, i.e. slot block_table[b][(ctx-1)/16] * 16 +
 * (ctx-1) % 16; then the ctx tokens, the new one included, are attended.
 * The page CTA whose share holds the new token's page quantises, writes and
 * attends it besides its cached pages (each unit's share of the page space
 * carries 96 pages without work after its last one, from 96 pages up, to
 * balance that), and the partials merge as in kvq_decode_attn_int2: the
 * cache bytes written are identical to kvq_append_int2's, and the output
 * equals that of the two calls in sequence up to the rounding order of the
 * merge.
 *   mu_k      device fp32 [H_kv][d], the key centre of the append
 *   cache     written at the new tokens' slots
 *   flags     0 or KVQ_STEP_INPUTS_READY
 *   other arguments as kvq_decode_attn_int2; kvq_decode_workspace_bytes(...,
 *   num_splits) covers this call.
 * With KVQ_STEP_INPUTS_READY the caller declares that R_k, R_v, mu_k,
 * block_table, context_lens and the cache are not written by the kernel
 * issued immediately before this call on the stream (in a model's decode
 * step that kernel is typically the projection that writes q, k_new and
 * v_new; the previous layer's step touches other caches): the kernel then
 * reads them, and starts streaming the cache, while that kernel finishes.
 * q, k_new, v_new, out and the workspace are always accessed after it.
 * Without the flag every input is read after it, as in every other call.
 * A sequence with ctx = 0 appends nothing and gets zeros; a new token whose
 * page id is outside [0, num_pages) is neither written nor attended, and
 * kvq_workspace_status reports KVQ_ERR_BAD_BLOCK_TABLE. */
enum { KVQ_STEP_INPUTS_READY = 1 };
kvq_status kvq_decode_step_int2(const void* q, const void* k_new, const void* v_new, int B, int H_q, int H_kv,
                                int d, void* cache, int64_t num_pages, const int32_t* block_table,
                                int max_pages_per_seq, const int32_t* context_lens, const float* mu_k,
                                const float* R_k, const float* R_v, float scale, float* out, void* workspace,
                                size_t workspace_bytes, int num_splits, int flags, void* stream);

/* Decode attention over the INT2 cache together with a BF16 window of
 * tokens kept unquantised.  "Output-Aware Rotation for INT2 KV-Cache
 * Quantization" §3.1 retains a small BF16 window; the Block-GTQ page keeps
 * 4 sink and 128 recent tokens in fp16 (Table 6).  The softmax runs over
 * the union of the context_lens[b] cached tokens and the first win_lens[b]
 * window tokens; a window token must not also be in the cached range (the
 * cached range need not start at the sequence's first token: keys are
 * stored after RoPE, so sinks and recent tokens can simply live in the
 * window).
 *   Arguments as kvq_decode_attn_int2, plus:
 *   mu_k      device fp32 [H_kv][d], the key centre append used: window
 *             logits are q . (k - mu_k) * scale, the same shift centring gives
 *             the cached keys
 *   win_k, win_v  device bf16 [B][win_max][H_kv][d], original basis (not
 *             centred, not rotated), 16-byte aligned
 *   win_lens  device int32 [B], clamped to [0, win_max]
 *   win_max   > 0
 * The window of each (sequence, KV head) is attended, after its cached pages,
 * by the page CTA whose share ends that unit (from 96 pages up each unit's
 * share of the page space carries win_max pages without work, at most
 * 256, after its last one, to balance that); the window's partial,
 * already in the output basis, is merged with the cache's as one more
 * split.  kvq_decode_workspace_bytes(..., num_splits) covers it. */
kvq_status kvq_decode_attn_int2_window(const void* q, int B, int H_q, int H_kv, int d,
                                       const void* cache, int64_t num_pages,
                                       const int32_t* block_table, int max_pages_per_seq,
                                       const int32_t* context_lens,
                                       const float* R_k, const float* R_v, const float* mu_k,
                                       const void* win_k, const void* win_v,
                                       const int32_t* win_lens, int win_max, float scale,
                                       float* out, void* workspace, size_t workspace_bytes,
                                       int num_splits, void* stream);

/* Reads (synchronously, on `stream`) and clears the error word a decode call
 * left in its workspace: KVQ_OK, KVQ_ERR_BAD_BLOCK_TABLE, or KVQ_ERR_CUDA
 * when an in-kernel wait gave up. */
kvq_status kvq_workspace_status(void* workspace, void* stream);

/* The same decode attention as kvq_decode_attn_int2, for callers that cannot
 * allocate device memory at call time: for example a serving loop whose
 * device memory is all planned once up front, a host application that owns
 * every device allocation through its own allocator, or code where the
 * device-wide synchronisation cudaMalloc may cause is not acceptable.  The
 * pages have no counterpart of this call; it is a packaging of the same
 * kernel.
 *   Arguments are those of kvq_decode_attn_int2 without the workspace.
 *   Scratch: a fixed 4 MiB array inside the library's device memory, held by
 *   every GPU that loads the library until the process exits.  A shape whose
 *   workspace (kvq_decode_workspace_bytes) exceeds 4 MiB is rejected with
 *   KVQ_ERR_WORKSPACE before anything is launched.
 *   The first call on a device looks up the array's device address (once
 *   per device, with that device current); make that first call before any
 *   stream capture.  Each call clears the scratch counters on `stream`.
 *   Every call shares the one array: calls whose work overlaps on the GPU
 *   (other streams, other host threads) race and give wrong results.
 *   Argument errors are returned before anything is enqueued.  No in-kernel
 *   error is reported (an out-of-range block-table entry, whose page is
 *   skipped, or a wait that ran out, which leaves the output partial): the
 *   scratch's error word is cleared by the next call and has no accessor.
 *   The array's address is looked up once per device, so the entry point
 *   must not be used across a cudaDeviceReset.  Allocates nothing. */
kvq_status kvq_decode_attn_int2_noalloc(const void* q, int B, int H_q, int H_kv, int d,
                                        const void* cache, int64_t num_pages,
                                        const int32_t* block_table, int max_pages_per_seq,
                                        const int32_t* context_lens,
                                        const float* R_k, const float* R_v, float scale,
                                        float* out, int num_splits, void* stream);

/* Test hook, not for production use: the next INT2 decode launch in this
 * process leaves the bulk copy of its first page unissued (the page's bytes
 * are still expected) and gives its waits a limit of about a millisecond, so
 * that wait runs out: the kernel records the timeout, lets its other copies
 * land, finishes without the missing page and returns, and
 * kvq_workspace_status then reports KVQ_ERR_CUDA.  Nothing faults or hangs;
 * the output of that call is incomplete. */
void kvq_debug_drop_next_copy(void);

/* ------------------------------------------------------------- Block-GTQ */

/* Host only.  Centroids (ascending, fp64) of the 2^b-level Lloyd-Max
 * quantiser of a standard Gaussian, 1 <= b <= 8, written to
 * centroids_out[0 .. 2^b).  The TQ-MSE scalar quantiser of an n-dimensional
 * sub-vector at width b uses fp32(c / sqrt(n)). */
kvq_status bgtq_lloyd_max_codebook(int b, double* centroids_out);

/* Block energy scores of a calibration prefix ("RoPE-Aware Bit Allocation
 * for KV-Cache Quantization", method step (1)): for KV head h and RoPE block
 * i = dims (i, i + d/2),
 *   scores[h][i] = 1/2 mean_{t < T, g in G(h)} ||q_{t,g}(i)||^2
 *                + 1/2 mean_{t < T} ||k_{t,h}(i)||^2,
 * G(h) the H_q/H_kv query heads reading KV head h (contiguous), and the
 * paired estimate (technical novelty (2): AM-GM gives paired <= scores)
 *   paired[h][i] = mean_{t, g in G(h)} ||q_{t,g}(i)|| ||k_{t,h}(i)||.
 *   q       device bf16 [T][H_q][d], post-RoPE calibration queries
 *   k       device bf16 [T][H_kv][d], post-RoPE calibration keys
 *   scores  device fp64 [H_kv][d/2], written (the input of bgtq_allocate)
 *   paired  device fp64 [H_kv][d/2] or null
 * Products of bf16 values are exact in fp64 and sums are fp64 (scores to
 * ~1e-15 relative); the paired estimate takes fp32 square roots (~1e-7
 * relative).  T = 0 gives zeros. */
kvq_status bgtq_energy_scores(const void* q, const void* k, int T, int H_q, int H_kv, int d,
                              double* scores, double* paired, void* stream);

/* Host only.  Greedy RoPE-block width allocation (Theorem 1): every block
 * starts at b_min; one bit at a time goes to the block with the largest
 * marginal gain (3/4) s_i 4^-b_i among blocks below b_max (ties: lowest
 * index), until sum(widths) == total_bits or every block is at b_max.
 *   scores      host fp64 [n_blocks], finite and >= 0
 *   widths_out  host int8 [n_blocks]
 * Requires 1 <= b_min <= b_max <= 8 and total_bits >= n_blocks * b_min. */
kvq_status bgtq_allocate(const double* scores, int n_blocks, int b_min, int b_max,
                         int64_t total_bits, int8_t* widths_out);

/* Bytes of one (page, KV head) Block-GTQ tile for a per-head key width
 * budget total_bits (sum over the 64 blocks) and value width v_bits:
 *   [0, 16*KB)          K codes, KB = 4*ceil(2*total_bits/32) bytes per slot:
 *                       LSB-first bit stream, groups by ascending width
 *                       1..8, each group's coordinates in order
 *   [16*KB, +256)       K norms, 8 fp16 per slot (entry b-1 = width-b group,
 *                       0 if that group is empty)
 *   [.., +16*VB)        V codes, VB = 16*v_bits: slot pair j (slots 2j,
 *                       2j+1) owns 2*VB bytes, an LSB-first stream of 128
 *                       channel entries of 2*v_bits bits, each the slot-2j
 *                       code then the slot-2j+1 code (one channel of two
 *                       tokens is one field: the decode's table index)
 *   [.., +32)           V norm, fp16 per slot
 * Returns 0 for unsupported arguments. */
size_t bgtq_tile_bytes(int total_bits, int v_bits);

/* Quantise-on-append into the Block-GTQ cache.
 *   k, v        device bf16 [n_tok][H_kv][d] (k post-RoPE)
 *   widths      device int8 [H_kv][d/2] per-block widths in 1..8 whose sum
 *               is at most total_bits (as bgtq_allocate returns them)
 *   pi_table    device fp32: shared orthogonal Pi_n (row-major n x n) for
 *               every even n <= d, Pi_n at pi_table + pi_offsets[n]
 *   pi_offsets  device int64 [d + 1] (-1 for odd n)
 *   codebooks   device fp64 [8][256]: row b-1 = bgtq_lloyd_max_codebook(b)
 * A slot's value codes share their pair row with the partner slot; the call
 * replaces only its own bits (atomically), so partners may be written in the
 * same call or in different ones.
 *   err_count   nullable device int32: incremented once per token whose slot
 *               lies outside [0, num_pages*16) (other than -1), and at least
 *               once when a head's widths are outside 1..8 or over budget;
 *               such tokens / heads are skipped
 * Key: RoPE block i = dims (i, i + d/2); blocks of equal width b form a
 * sub-vector (ascending block index, each block as its two dims) of length
 * n; r = ||x|| (fp32 fma chain of squares, correctly rounded sqrt),
 * u = x / r, y = u Pi_n (fp32 fma chain), code = nearest of
 * fp32(c_b / sqrt(n)) (ties to the lower index), norm = fp16(r).
 * Value: the same with n = d and width v_bits. */
kvq_status bgtq_append(const void* k, const void* v, int n_tok, int H_kv, int d,
                       const int32_t* slot_mapping, const int8_t* widths, int total_bits,
                       int v_bits, const float* pi_table, const int64_t* pi_offsets,
                       const double* codebooks, void* cache, int64_t num_pages,
                       int32_t* err_count, void* stream);

/* Fused packed-cache decode attention over the Block-GTQ cache; arguments as
 * kvq_decode_attn_int2 plus the format parameters of bgtq_append.  Logits
 * are <q, k^>*scale with k^ the decoded post-RoPE key; out = softmax . V^.
 * q, cache and workspace must be 16-byte aligned (KVQ_ERR_INVALID_ARG
 * otherwise).  The scaled centroids the decode multiplies by are
 * fp32(C_b[c] * (1/sqrt(n))) with the reciprocal in fp64: equal to the
 * append's fp32(C_b[c] / sqrt(n)) but for a rare last-bit difference, which
 * only moves a logit by an fp32 rounding. */
kvq_status bgtq_decode_attn(const void* q, int B, int H_q, int H_kv, int d,
                            const void* cache, int64_t num_pages,
                            const int32_t* block_table, int max_pages_per_seq,
                            const int32_t* context_lens,
                            const int8_t* widths, int total_bits, int v_bits,
                            const float* pi_table, const int64_t* pi_offsets,
                            const double* codebooks, float scale,
                            float* out, void* workspace, size_t workspace_bytes,
                            int num_splits, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
