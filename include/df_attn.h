/*
 * df_attn.h -- C ABI of the GB300 (sm_103a) exact DeBERTa-v2/v3 disentangled
 * self-attention library (libdfattn.so): forward and fused backward, computed
 * without ever storing the [B, H, L, L] score matrix.
 *
 * The operation (per sequence, per head h; tokens i, j counted inside the
 * sequence; R = 2 * att_span):
 *
 *   delta(i, j) = clamp(bucket(i - j) + att_span, 0, R - 1)
 *   S[i, j]     = c * (Q_i.K_j + Q_i.Kr[delta] + K_j.Qr[delta])     c = 1/sqrt(3D)
 *   P           = softmax_j(S) with -inf for masked queries / keys
 *   O           = (P * keep / (1 - p)) V ;   LSE_i = log sum_j exp(S[i, j])
 *
 * bucket() is DeBERTa's log bucketing: |r| <= nb/2 keeps r, larger |r| maps
 * to sign(r) * (nb/2 + ceil(ln(|r| / (nb/2)) / ln((mp - 1) / (nb/2)) * (nb/2 - 1)))
 * (nb = position_buckets, mp = max_relative_positions; no bucketing when
 * either is <= 0).
 *
 * Passages this follows -- "DisentangledFlash" (pypi disentangled-flash
 * 1.1.1): section "Status" (exact C2P/P2C DeBERTa-v2/v3 attention without the
 * [B, H, L, L] matrix, FP16 / BF16 / strict FP32, head dims 32/64/128,
 * factorised 2-D padding masks, lengths up to 8192, packed cu_seqlens
 * training, Philox dropout regenerated in backward); section "Hugging Face
 * usage" (an LSE-producing training forward, a dQ kernel and a dK/dV kernel);
 * section "Performance" (the relative-position products over R rows and the
 * relative-position gradients counted in the FLOP formula).
 *
 * Conventions shared by every entry point
 *   - All tensors are dense and contiguous; the caller owns every buffer.
 *     No entry point allocates device memory; scratch comes from the
 *     caller's workspace (size from df_attn_workspace_size), except for
 *     df_attn_fwd_noalloc, whose scratch is an 8 MiB static device array of
 *     the library (held on every GPU that loads it).
 *   - Device pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *   - Argument errors return a status before anything is enqueued and
 *     nothing is written.  There is no fallback path: an unsupported
 *     configuration returns DF_ERR_UNSUPPORTED.  No C++ exception crosses
 *     this boundary.
 *   - Errors found on the device (inconsistent cu_seqlens, a bounded wait
 *     that gave up) are recorded in the workspace and reported by
 *     df_get_device_error.
 */
#ifndef DF_ATTN_H
#define DF_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same type as cudaStream_t). */
typedef struct CUstream_st *df_stream_t;

typedef enum {
    DF_OK = 0,
    DF_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or value      */
    DF_ERR_UNSUPPORTED = 2,   /* valid but outside the supported contract   */
    DF_ERR_WORKSPACE = 3,     /* workspace missing or too small             */
    DF_ERR_CUDA = 4,          /* a CUDA runtime / launch error              */
    DF_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up         */
    DF_ERR_DEVICE_ARG = 6,    /* the device found inconsistent cu_seqlens   */
    DF_ERR_DEVICE_CHECK = 7   /* checked build: an index outside its buffer */
} df_status;

typedef enum {
    DF_BF16 = 0,              /* bf16 storage, fp32 accumulation (tensor cores) */
    DF_FP16 = 1,              /* fp16 storage, fp32 accumulation (tensor cores) */
    DF_FP32 = 2,              /* strict fp32 (CUDA-core fp32 arithmetic)        */
    DF_FP32_FAST = 3          /* fp32 storage, fast mode (below)                */
} df_dtype;

/*
 * Fast fp32 mode (DF_FP32_FAST; "DisentangledFlash", section "Status": an
 * optional fast FP32/TF32 mode beside the strict fp32 one).  Every tensor is
 * fp32 as for DF_FP32, the LSE fp32 as always.  The inputs are rounded to
 * nearest fp16 -- the same 10-bit significand as TF32 -- in the workspace,
 * the fp16 tensor-core kernels run on them (fp32 accumulation, 16-bit P and
 * dZ as for DF_FP16), and O and the gradients come back widened to fp32 from
 * their fp16 results.  Error: that of DF_FP16 plus the input rounding
 * (relative 2^-11 per element); tensors must stay within the fp16 range
 * (|x| < 65504, else inf / NaN results).  Same contract as DF_FP16 otherwise
 * (saved band bias included); the workspace adds the fp16 copies of the
 * inputs and outputs.
 */

/*
 * Problem description.
 *   Padded layout (cu_seqlens == NULL): B sequences of L tokens; Q, K, V, O,
 *     dO, dQ, dK, dV are [B, L, H, D]; LSE is fp32 [B, H, L].
 *   Packed layout (cu_seqlens != NULL): B sequences back to back,
 *     cu_seqlens[0] = 0, cu_seqlens[b+1] - cu_seqlens[b] = length of
 *     sequence b (1 <= length <= L, L = the longest length),
 *     cu_seqlens[B] = total_tokens; tensors are [total_tokens, H, D]; LSE is
 *     fp32 [H, total_tokens].  No padding token is computed.
 *   Qr, Kr, dQr, dKr are [H, R, D] with R = 2 * att_span.
 *   query_mask / key_mask: padded layout only, [B, L] bytes (0 = masked),
 *     or NULL.  The 2-D mask is query_mask (x) key_mask.  A row with no
 *     attendable key (masked query, or all keys masked) gets O = 0,
 *     LSE = +inf and zero gradients.
 *   Dropout of the attention probabilities (dropout_p in [0, 1)): keep[i,j]
 *     is word (j & 3) of Philox4x32-10(counter = (j >> 2, i, b*H + h,
 *     philox_offset), key = (seed low 32 bits, seed high 32 bits)) compared
 *     with floor((1 - dropout_p) * 2^32); i, j are positions inside the
 *     sequence.  The mask is regenerated in the backward, never stored.
 *     philox_offset must be < 2^32.
 *   softmax_scale: c; 0 selects 1/sqrt(3D).
 */
typedef struct {
    int32_t B, L, H, D;
    const int32_t *cu_seqlens;     /* device [B+1] int32, or NULL (padded)   */
    int32_t total_tokens;          /* packed layout only                      */
    int32_t att_span;              /* R = 2 * att_span relative rows          */
    int32_t position_buckets;      /* nb (<= 0: no log bucketing)             */
    int32_t max_relative_positions;/* mp (<= 0: no log bucketing)             */
    const uint8_t *query_mask;     /* device [B, L] or NULL (padded only)     */
    const uint8_t *key_mask;       /* device [B, L] or NULL (padded only)     */
    float dropout_p;
    uint64_t philox_seed;
    uint64_t philox_offset;
    float softmax_scale;
    df_dtype dtype;
    void *band_bias;               /* saved band bias (device) or NULL; below */
} df_attn_params;

/*
 * Supported contract: D in {32, 64, 128}; 1 <= L <= 8192; 1 <= att_span <=
 * 512; B, H >= 1 and B * L * H < 2^31 (padded) or total_tokens * H < 2^31
 * (packed); when log bucketing is on, position_buckets >= 2 and
 * max_relative_positions - 1 > position_buckets / 2, and for bf16 / fp16
 * also (m - 1) ln(1 + 1/m) <= ln((max_relative_positions - 1) / m) with
 * m = position_buckets / 2 (the bucketed index then moves by at most one per
 * relative position; e.g. 256 buckets need max_relative_positions >= 345).
 */

/*
 * Saved band bias (bf16 / fp16 / fast fp32; ignored for DF_FP32).  Near the
 * diagonal every (query, key) pair has its own relative-position term
 * c log2(e) (Q_i . Kr[delta] + K_j . Qr[delta]) ("DisentangledFlash",
 * section "Status": C2P and P2C).  The backward needs it again for every
 * band tile.  With p->band_bias == NULL the backward recomputes it into its
 * workspace; with a device buffer of df_attn_band_bias_size(p) bytes
 * (16-byte aligned, caller-owned) df_attn_fwd writes it there as a by-product
 * and df_attn_bwd reads it from there, like the LSE: the backward must then
 * get the same buffer, unchanged since the forward with the same inputs and
 * parameters.  Layout: fp16 128 x 128 blocks of 128-query x 128-key pairs,
 * base-2 units, kept for the key blocks within a fixed reach of each query
 * block (private to the library).  0 for invalid parameters or DF_FP32.
 */
size_t df_attn_band_bias_size(const df_attn_params *p);

/* Bytes of device workspace that df_attn_fwd (backward = 0) or df_attn_bwd
 * (backward != 0) needs for these parameters; 0 if the parameters are
 * invalid.  The workspace holds the relative-index table, per-token
 * relative-position dot products, the device error word and, for the
 * backward, the row terms Dl_i, the diagonal sums of dZ used for the
 * relative-position gradients ([T, H, R] twice, in the input dtype for bf16 /
 * fp16 and fp32 for strict fp32), fp32 partial sums of dQr / dKr and, for
 * bf16 / fp16 when p->band_bias is NULL, the band bias.  DF_FP32_FAST: the
 * fp16 workspace followed by fp16 copies of the inputs and outputs (forward:
 * Q, K, V, Qr, Kr, O; backward also dO, dQ, dK, dV, dQr, dKr). */
size_t df_attn_workspace_size(const df_attn_params *p, int backward);

/*
 * Forward.  Writes out (same dtype and layout as q) and lse (fp32, natural
 * log, layout above; +inf for rows with no attendable key).
 * q, k, v: [B, L, H, D] or [T, H, D] in p->dtype; qr, kr: [H, R, D].
 */
df_status df_attn_fwd(const df_attn_params *p, const void *q, const void *k, const void *v, const void *qr,
                      const void *kr, void *out, float *lse, void *workspace, size_t workspace_bytes,
                      df_stream_t stream);

/*
 * Inference forward: the same output as df_attn_fwd without the row
 * log-sum-exp, which only the backward needs ("DisentangledFlash", section
 * "Status": an inference path beside the training path; section "Hugging
 * Face usage": the training forward is the LSE-producing one).  Same
 * arguments, workspace (df_attn_workspace_size(p, 0)) and errors as
 * df_attn_fwd, minus lse.
 */
df_status df_attn_fwd_inference(const df_attn_params *p, const void *q, const void *k, const void *v,
                                const void *qr, const void *kr, void *out, void *workspace, size_t workspace_bytes,
                                df_stream_t stream);

/*
 * Backward.  Takes the forward's inputs, its out and lse, and dout (layout of
 * out); writes dq, dk, dv (layout of q) and dqr, dkr ([H, R, D], summed over
 * the batch, overwritten).  All gradients are deterministic: the same call
 * gives bitwise the same results (no floating-point atomics; relative-
 * position gradients are reduced in a fixed order).
 * Ordering: the work is ordered after earlier work on `stream` and later
 * work on `stream` waits for all of it.  Internally the dQ kernel runs on a
 * per-device side stream (created on the first backward on that device)
 * forked from `stream` by an event and joined back before the call's last
 * kernels, so that it overlaps the dK/dV kernel.
 */
df_status df_attn_bwd(const df_attn_params *p, const void *q, const void *k, const void *v, const void *qr,
                      const void *kr, const void *out, const float *lse, const void *dout, void *dq, void *dk,
                      void *dv, void *dqr, void *dkr, void *workspace, size_t workspace_bytes,
                      df_stream_t stream);

/*
 * One training step of the layer from HOST buffers: copies q, k, v, qr, kr,
 * dout from host memory to the device arena, runs the forward and the
 * backward, and copies out, lse, dq, dk, dv, dqr, dkr back to host memory,
 * all on `stream`; returns after the stream has finished.  In this call
 * p->cu_seqlens, p->query_mask and p->key_mask are HOST pointers (copied
 * too).  Host buffers should be pinned for full copy bandwidth.  The device
 * arena (caller-owned, df_attn_step_host_arena_size bytes) holds the device
 * copies, the band bias the forward saves for the backward and the
 * workspace.  A per-device copy stream (created on the first call on that
 * device) overlaps the copies with the kernels: with B >= 2 (16-bit dtypes)
 * the forward runs in two parts, the first half of the sequences' q, k, v
 * going up on `stream` and the rest on the copy stream while the first part
 * runs; dout goes up while the forward runs; out and lse come down while the
 * backward runs, dq, dv and dk each once it is final, while the remaining
 * kernels run.
 */
size_t df_attn_step_host_arena_size(const df_attn_params *p);
df_status df_attn_step_host(const df_attn_params *p, const void *q, const void *k, const void *v, const void *qr,
                            const void *kr, const void *dout, void *out, float *lse, void *dq, void *dk, void *dv,
                            void *dqr, void *dkr, void *device_arena, size_t arena_bytes, df_stream_t stream);

/*
 * Forward that allocates nothing (the paper has no counterpart; this is a
 * deployment convenience).  For callers that cannot allocate device memory
 * -- code inside a host framework that owns all device memory (a plugin or
 * custom operator whose allocator it may not grow), or latency-critical
 * loops where cudaMalloc's implicit synchronisation is not acceptable.  Same
 * arguments and results as df_attn_fwd minus the workspace: the scratch lives
 * in a file-scope device array of 8 MiB that every GPU loading this library
 * holds until the process exits.  The caller still passes inputs and outputs.
 *   - Limit: df_attn_workspace_size(p, 0) <= 8 MiB, i.e. about
 *     16 * total_tokens * H + 8 * L bytes (e.g. 16,384 tokens x 24 heads);
 *     larger problems return DF_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and give undefined results; serialise them.
 *   - Device-side errors (inconsistent cu_seqlens, a give-up) land in the
 *     array's error word: df_attn_fwd_noalloc_device_error reads it.
 *   - The cached address assumes the device's primary context, which is what
 *     the CUDA runtime uses; it is not valid after cudaDeviceReset.
 */
df_status df_attn_fwd_noalloc(const df_attn_params *p, const void *q, const void *k, const void *v,
                              const void *qr, const void *kr, void *out, float *lse, df_stream_t stream);

/* Synchronises `stream` and reads the device error word of the static
 * scratch used by df_attn_fwd_noalloc on the current device (see
 * df_get_device_error); DF_OK before the first such call. */
df_status df_attn_fwd_noalloc_device_error(df_stream_t stream);

/*
 * Packing ("DisentangledFlash", section "Packed unpadded inference and
 * training": pack_padded_with_info / unpack_packed).  A padded batch of B
 * sequences of L positions with a padding mask [B, L] (device bytes, 0 =
 * padding) becomes the packed layout: the valid positions of each sequence in
 * order, sequence after sequence; a sequence without any valid position is
 * dropped.  With right padding (every sequence's valid positions first),
 * attention over the packed layout equals the masked padded attention on the
 * valid rows; other masks move positions, and with them relative positions.
 *
 * df_pack_info writes, on the device and asynchronously on `stream`:
 *   cu_seqlens [B + 1] int32: offsets of the non-empty sequences (the first
 *     info[2] + 1 entries are used);
 *   index [B * L] int32: index[t] = b * L + l, the padded row of packed row t
 *     (the first info[0] entries are used);
 *   info [3] int32: total packed tokens, longest sequence, non-empty sequences
 *     (read it back for the attention's total_tokens, L and B).
 * workspace: df_pack_workspace_size(B) bytes, 4-byte aligned.
 *
 * df_pack_rows: packed[t] = padded[index[t]] for t < min(info[0], max_rows),
 *   rows of row_bytes bytes (a multiple of 16, both buffers 16-byte aligned);
 *   padded has padded_rows rows (an index outside them gives a zero row).
 * df_unpack_rows: padded[index[t]] = packed[t] for t < min(info[0],
 *   max_rows); every other of the padded_rows rows is zero.
 * All three are deterministic (no atomics on the data).
 */
size_t df_pack_workspace_size(int32_t B);
df_status df_pack_info(const uint8_t *mask, int32_t B, int32_t L, int32_t *cu_seqlens, int32_t *index,
                       int32_t *info, void *workspace, size_t workspace_bytes, df_stream_t stream);
df_status df_pack_rows(const void *padded, int32_t padded_rows, const int32_t *index, const int32_t *info,
                       int32_t max_rows, size_t row_bytes, void *packed, df_stream_t stream);
df_status df_unpack_rows(const void *packed, const int32_t *index, const int32_t *info, int32_t max_rows,
                         size_t row_bytes, int32_t padded_rows, void *padded, df_stream_t stream);

/*
 * The steps on either side of the attention ("DisentangledFlash", section
 * "Status": the fused QKV projection is always on; section "Hugging Face
 * usage": the query / key / value and relative-position projections stay in
 * the autograd graph).  DeBERTa-v2/v3 with shared attention keys: one weight
 * w = [W_q; W_k; W_v] ([3, H*D, C], row-major, rows of head h at h*D) and
 * bias b = [b_q; b_k; b_v] ([3, H*D], or NULL) project the hidden states, and
 * W_q, W_k with b_q, b_k also project the layer-normalised relative
 * embeddings.  bf16 / fp16 storage, fp32 accumulation (cuBLASLt products
 * without workspace, small kernels for the layer norm and the sums, which
 * run in a fixed order).  Device pointers 16-byte aligned; C, H*D and D
 * multiples of 8.  Nothing is allocated.
 *
 * df_qkv_proj_fwd: qkv [3, T, H*D] = x [T, C] W_j^T + b_j for j = q, k, v (Q,
 *   K, V back to back, each in the [T, H, D] layout of df_attn_fwd).
 * df_qkv_proj_bwd: from dqkv [3, T, H*D]: dx [T, C] = sum_j dY_j W_j (j in
 *   order); dw [3, H*D, C] (+)= dY_j^T x; dbias [3, H*D] (+)= sum_t dY_j[t]
 *   (skipped when NULL; then the workspace may be NULL); `accumulate` != 0
 *   adds to dw / dbias.  workspace: df_qkv_proj_workspace_size(H*D) bytes
 *   (fp32 partial column sums).
 * df_rel_proj_fwd: rel_ln [R, C] = LayerNorm(rel [R, C]; gamma, beta, eps)
 *   (kept for the backward, with ln_stats [R, 2] fp32 = mean, 1/std);
 *   qr[h] = rel_ln W_q[h]^T + b_q[h], kr[h] = rel_ln W_k[h]^T + b_k[h] ([H, R,
 *   D], the layout of df_attn_fwd).  rel holds the R = 2 * att_span rows of
 *   the relative-embedding table the attention uses.
 * df_rel_proj_bwd: from dqr, dkr [H, R, D]: drel [R, C]; dgamma, dbeta [C];
 *   rows q and k of dw [3, H*D, C] and of dbias [3, H*D] (NULL: skipped);
 *   `accumulate` != 0 adds to dgamma, dbeta, dw and dbias (after
 *   df_qkv_proj_bwd, for the shared weights).  workspace:
 *   df_rel_proj_workspace_size bytes.
 */
df_status df_qkv_proj_fwd(int32_t T, int32_t C, int32_t HD, df_dtype dtype, const void *x, const void *w,
                          const void *bias, void *qkv, df_stream_t stream);
size_t df_qkv_proj_workspace_size(int32_t HD);
df_status df_qkv_proj_bwd(int32_t T, int32_t C, int32_t HD, df_dtype dtype, const void *x, const void *w,
                          const void *dqkv, void *dx, void *dw, void *dbias, int32_t accumulate, void *workspace,
                          size_t workspace_bytes, df_stream_t stream);
size_t df_rel_proj_workspace_size(int32_t R, int32_t C, int32_t H, int32_t D);
df_status df_rel_proj_fwd(int32_t R, int32_t C, int32_t H, int32_t D, df_dtype dtype, const void *rel,
                          const void *gamma, const void *beta, float eps, const void *w, const void *bias,
                          void *rel_ln, float *ln_stats, void *qr, void *kr, df_stream_t stream);
df_status df_rel_proj_bwd(int32_t R, int32_t C, int32_t H, int32_t D, df_dtype dtype, const void *rel,
                          const void *gamma, const void *rel_ln, const float *ln_stats, const void *w,
                          const void *dqr, const void *dkr, void *drel, void *dgamma, void *dbeta, void *dw,
                          void *dbias, int32_t accumulate, void *workspace, size_t workspace_bytes,
                          df_stream_t stream);

/*
 * The relative-position index table delta(r) for r = -(L-1) .. L-1, written
 * as int32 to out_dev[r + L - 1] (device, 2L - 1 entries), computed on the
 * device exactly as the attention kernels use it.  For bit-exact checks.
 */
df_status df_rel_index_table(int32_t L, int32_t att_span, int32_t position_buckets,
                             int32_t max_relative_positions, int32_t *out_dev, df_stream_t stream);

/*
 * The dropout keep mask of sequence b, head h, drawn on the device by the
 * same generator code as the attention kernels ("DisentangledFlash",
 * section "Status": the Philox mask is regenerated in the backward, never
 * stored -- this entry point exists so that tests can compare it bit for bit
 * with an independent generator).  form 0: the row generator of the forward
 * and dQ kernels; form 1: the column generator of the dK/dV kernel.  Writes
 * out_dev[i * n + j] = keep(i, j) (0 / 1 bytes, device, n * n bytes, n = the
 * length of sequence b: L padded, cu_seqlens[b+1] - cu_seqlens[b] packed).
 * Uses p's dropout_p, philox_seed, philox_offset, H and layout.
 */
df_status df_dropout_keep_mask(const df_attn_params *p, int32_t b, int32_t h, int32_t form, uint8_t *out_dev,
                               df_stream_t stream);

/*
 * Synchronises `stream` and reads the device error word of a workspace that
 * was passed to df_attn_fwd / df_attn_bwd: DF_OK, DF_ERR_DEVICE_ARG
 * (cu_seqlens inconsistent with B, L, total_tokens), DF_ERR_TIMEOUT (a
 * bounded device wait gave up; the affected outputs are unspecified) or, in
 * a library built with DF_CHECKED (exact_deberta_disentangled_gb300.build,
 * checked=True), DF_ERR_DEVICE_CHECK: a shared-memory gather or window copy
 * of a tensor-core kernel computed an index outside its buffer (the access
 * was clamped into range; the outputs are unspecified).  The
 * word is cleared at the start of every df_attn_fwd / df_attn_bwd call.
 */
df_status df_get_device_error(const void *workspace, df_stream_t stream);

/*
 * Benchmark timing hooks.  `events` holds 8 CUDA event handles (cudaEvent_t,
 * created by the caller, on the device the calls run on): while set, every
 * df_attn_fwd / df_attn_bwd records events[2k] just before and events[2k+1]
 * just after kernel phase k on the call's stream -- k = 0 the forward
 * attention kernel, 1 the dQ kernel, 2 the dK/dV kernel, 3 the relative-
 * position gradient kernels.  Pass NULL / 0 to switch the hooks off.  The
 * setting is process-wide and not thread-safe; it exists for measurement only.
 */
df_status df_attn_set_profile_events(void *const *events, int n);

/*
 * Test hook for the bounded-wait path (process-wide, not thread-safe).  From
 * the next call on, the MMA-issuing warp of every CTA of one attention kernel
 * (kernel 0 = forward, 1 = dQ, 2 = dK/dV) stops issuing when it reaches tile
 * `tile` of its loop, and every device wait gives up once wait_limit_ns
 * (at most 2 s) have passed and wait_min_probes probes have failed.  The
 * kernel's other roles then wait for work that never comes, give up, record
 * DF_ERR_TIMEOUT (read it with df_get_device_error) and leave the kernel:
 * the outputs of such a call are unspecified and the CUDA context stays
 * usable.  kernel = -1 switches the injection off and restores the default
 * limits (2 s and 2^20 probes).  Nothing else uses it.
 */
df_status df_attn_debug_inject_stall(int kernel, int tile, uint64_t wait_limit_ns, uint32_t wait_min_probes);

/* Static, human-readable name of a status code. */
const char *df_status_string(df_status s);

/* Library version, "major.minor.patch". */
const char *df_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DF_ATTN_H */
