/*
 * attn.h -- C ABI of the GB300 fused-attention library (libattn_gb300.so).
 *
 * Scaled-dot-product attention with tiled online softmax on one GPU:
 * forward with saved log-sum-exp, FlashAttention-2-style backward, and
 * split-KV decode for a short query block over a long KV cache.
 *
 * What is computed (per batch b, query head h, query row i, key j):
 *   kv     = h / (H / Hkv)      consecutive query heads share a KV head
 *          (brotensor ops/flash_attention.h, flash_attention_decode: query head h
 *           maps to KV head h/(num_q_heads/num_kv_heads))
 *   p      = i + q_offset       absolute query position
 *          (ferrotensor_backend engine/attention.rs, AttentionOptions.causal_offset)
 *   s      = scale * q_i . k_j
 *   st     = softcap > 0 ? softcap * tanh(s / softcap) : s
 *          (brotensor ops/flash_attention.h, flash_attention_decode, Gemma-2
 *           extensions: after the scale, before mask and softmax; 0 = off)
 *   key j visible iff  (!causal || j <= p)
 *                   && (window == 0 || |p - j| < window)
 *                   && (key_mask == NULL || key_mask[b*stride + j] > 0.5)
 *          (ferrotensor AttentionOptions for causal/window -- with causal this is
 *           keys [max(0, p-window+1), p] as brotensor flash_attention_decode and
 *           forge attention.metal AttnParams state; brotensor flash_attention_backward
 *           for the 1/0 key mask with the 0.5 threshold)
 *   O_i    = sum_j softmax_j(st_ij over visible j) v_j
 *   LSE_i  = ln sum_{visible j} exp(st_ij)      natural log, capped scores
 *          (vision_rs flash_attn2.rs, Forward: logsumexp saved for backward)
 *   A row with no visible key gets O_i = 0 and LSE_i = -inf and adds nothing to
 *   any gradient.
 *
 * Layouts (all row-major, contiguous, caller-owned device memory):
 *   q, o, do, dq : [B][Tq][H*hd]     k, v, dk, dv : [B][Tk][Hkv*hd]
 *   lse          : [B][H][Tq] fp32
 *   key_mask     : fp32, key j of batch b at key_mask[b*key_mask_bstride + j];
 *                  key_mask_bstride = 0 shares one length-Tk mask across batches.
 *   (forge attention.metal: q/o [B,T,H*hd], k/v [B,T,Hkv*hd]; brotensor: a
 *    length-Lk fp32 key mask, caller-owned.)
 *
 * Ownership and execution: the library never allocates, frees or synchronises.
 * Every call validates its arguments on the host, then enqueues kernels on
 * `stream` (a cudaStream_t passed as void*; NULL = legacy default stream) and
 * returns.  Outputs and gradients are overwritten, never accumulated
 * (ferrotensor engine/attention.rs, flash_attention_backward: gradients are
 * stored over the buffers' contents).
 * Pointers must be 16-byte aligned.  The device current on the calling thread
 * must own every pointer.
 *
 * Errors: argument errors return ATTN_ERR_INVALID_ARG (or ATTN_ERR_UNSUPPORTED
 * for a valid but unimplemented shape/dtype) before anything is enqueued and
 * nothing is written.  A failed launch returns ATTN_ERR_CUDA.  Kernels never
 * trap: every wait inside a kernel is bounded, and a wait that runs out sets a
 * device status word that attn_get_device_status() reports as ATTN_ERR_TIMEOUT.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,
    ATTN_ERR_UNSUPPORTED = 2,
    ATTN_ERR_CUDA = 3,
    ATTN_ERR_TIMEOUT = 4
} attn_status;

typedef enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 } attn_dtype;

/*
 * Forward.  O = softmax(st) V over the visible keys, LSE saved when lse != NULL.
 * Source: vision_rs flash_attn2.rs, Forward (online softmax with saved
 * logsumexp); ferrotensor flash_attention_v2_with (GQA, causal offset, window);
 * brotensor flash_attention_gqa_forward / flash_attention_windowed_forward
 * (key mask, softcap, bidirectional encoder case).
 *   dt        : element type of q, k, v, o (fp32 math inside for every type).
 *   q, k, v   : inputs, layouts above.          o : output [B][Tq][H*hd].
 *   lse       : output [B][H][Tq] fp32, or NULL to skip.
 *   B, Tq, Tk : batch, query rows, key rows (>= 0; B or Tq == 0 is a no-op,
 *               Tk == 0 writes O = 0, LSE = -inf).
 *   H, Hkv    : query / KV heads, Hkv >= 1 divides H.
 *   hd        : head dim 32, 64, 96, 128 or 256.  16-bit types run on the tensor
 *               cores (32 and 96 as 64 and 128 with the columns past the head read as
 *               zeros; 256 with one 128-row query tile per work item; with an additive
 *               bias, or in packed sequences, 32, 96 and 256 take the CUDA-core
 *               kernels); fp32 runs on CUDA-core kernels (same results, no tensor-core
 *               speed).  attn_bwd at hd 256 (dense, no bias) runs on the tensor cores
 *               in separate dV, dK and dQ passes.
 *   scale     : > 0 and finite (1/sqrt(hd) in the usual case).
 *   causal    : 0/1.   window : >= 0, 0 = unbounded.   softcap : >= 0, 0 = off.
 *   q_offset  : >= 0, absolute position of query row 0.
 *   key_mask  : NULL or fp32 mask as above; key_mask_bstride >= 0.
 */
ATTN_API attn_status attn_fwd(attn_dtype dt, const void* q, const void* k, const void* v, void* o,
                     float* lse, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale,
                     int causal, int window, float softcap, int q_offset, const float* key_mask,
                     long long key_mask_bstride, void* stream);

/* Bytes of scratch attn_bwd needs: -D = -rowsum(dO * O) and -LSE*log2(e), one
 * fp32 each per (b, h, i), rows padded to a multiple of 64 queries (D is forge
 * attention.metal's attention_bwd_d_f32 quantity).  Host only; 0 for B, Tq or H
 * below 1. */
ATTN_API size_t attn_bwd_workspace_size(int B, int Tq, int H);

/*
 * Backward (FlashAttention-2 style, deterministic, no atomics).
 * Source: vision_rs flash_attn2.rs, "Backward - dQ" and "Backward - dK / dV";
 * forge attention.metal, attention_bwd_d_f32 (D = dO.O), attention_bwd_dq_f32,
 * attention_bwd_dkv_f32 (softcap derivative 1 - tanh^2, GQA group sums);
 * ferrotensor flash_attention_v2_backward_with (separate dQ and dK/dV passes).
 *   o, lse    : the forward's output and saved LSE for the same arguments.
 *   dout      : upstream gradient of o, layout of q.
 *   dq, dk, dv: outputs, layouts of q, k, v; overwritten.
 *   workspace : device scratch of at least attn_bwd_workspace_size() bytes,
 *               16-byte aligned; contents on entry are ignored.
 *   Other arguments exactly as for attn_fwd (same values as the forward call).
 */
ATTN_API attn_status attn_bwd(attn_dtype dt, const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, int B, int Tq, int Tk, int H,
                     int Hkv, int hd, float scale, int causal, int window, float softcap,
                     int q_offset, const float* key_mask, long long key_mask_bstride,
                     void* stream);

/*
 * The three passes of attn_bwd, selectable one at a time (same arguments).
 * Source: ferrotensor engine/attention.rs, flash_attention_v2_backward_with (a
 * dQ dispatch over query tiles and a dK/dV dispatch over key tiles); forge
 * attention.metal, attention_bwd_d_f32 (the D pass).
 * phases is a bit set: 1 = D = rowsum(dO*O) and LSE*log2(e) into the
 * workspace (stored negated), 2 = dK/dV, 4 = dQ.  Pass 4 forms D and LSE*log2(e) itself and
 * leaves them in the workspace (so with 4 set, 1 is implied and, on the
 * 16-bit path, not run as a pass of its own); pass 2 alone reads the workspace
 * an earlier pass 1 or 4 with the same arguments wrote.  Requested passes run
 * as 1, 4, 2.  attn_bwd(...) is attn_bwd_phases(..., 7).
 */
ATTN_API attn_status attn_bwd_phases(attn_dtype dt, const void* q, const void* k, const void* v,
                     const void* o, const void* dout, const float* lse, void* dq, void* dk,
                     void* dv, void* workspace, size_t workspace_bytes, int B, int Tq, int Tk,
                     int H, int Hkv, int hd, float scale, int causal, int window, float softcap,
                     int q_offset, const float* key_mask, long long key_mask_bstride,
                     void* stream, int phases);

/* Bytes of scratch attn_decode needs (split-KV partials); 0 if the shape is invalid. */
ATTN_API size_t attn_decode_workspace_size(int B, int Lq, int Tk, int H, int Hkv, int hd);

/*
 * The key split attn_decode, attn_decode_len (with Tk = the capacity) and
 * attn_decode_noalloc use for a shape: the cache rows [0, Tk) fall into
 * *splits chunks of *chunk rows (a multiple of 64; the last chunk may be
 * shorter), one CTA per (b, KV head, 16 query rows of the group, chunk).  The
 * split is a deterministic function of the shape (it changes only the
 * rounding of the result: brotensor ops/flash_attention.h,
 * flash_attention_decode_len).  Host only, no CUDA call.  Returns
 * ATTN_ERR_INVALID_ARG (outputs untouched) when a pointer is NULL, B, Lq, H or
 * Hkv is not positive, Tk is negative or Hkv does not divide H.
 */
ATTN_API attn_status attn_decode_plan(int B, int Lq, int Tk, int H, int Hkv, int* splits, int* chunk);

/*
 * Split-KV decode: a block of Lq query rows (1 <= Lq <= 16) at positions
 * q_offset .. q_offset+Lq-1 over a KV cache of Tk rows.  Each (b, KV head,
 * key chunk) is one CTA that reads its K/V rows once for all (H/Hkv)*Lq query
 * rows of the group; a second kernel merges the chunks by log-sum-exp.
 * Source: brotensor ops/flash_attention.h, flash_attention_decode (query p =
 * valid_len - L_q + q attends [0, p], GQA, softcap, window) and
 * flash_attention_decode_len (work divided over the keys; split points change
 * only the rounding; R > 1 rows each read the cache once).
 *   dt        : ATTN_BF16 or ATTN_F16 (ATTN_F32 runs the fp32 forward kernel).
 *   q, o      : [B][Lq][H*hd];  k, v : [B][Tk][Hkv*hd];  lse : [B][H][Lq] or NULL.
 *   workspace : device scratch of at least attn_decode_workspace_size() bytes,
 *               16-byte aligned.
 *   (H/Hkv)*Lq <= 64; 16-bit types take hd 64, 128 or 256 (the split kernel's
 *   sizes), fp32 any attn_fwd head size; the rest as for attn_fwd.  The usual KV-cache call is causal with q_offset =
 *   Tk - Lq.
 */
ATTN_API attn_status attn_decode(attn_dtype dt, const void* q, const void* k, const void* v, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, int B, int Lq,
                        int Tk, int H, int Hkv, int hd, float scale, int causal, int window,
                        float softcap, int q_offset, const float* key_mask,
                        long long key_mask_bstride, void* stream);

/*
 * Split-KV decode over a fixed-capacity KV cache whose valid length per
 * sequence lives in device memory, so that a captured CUDA graph can be
 * replayed as the cache grows without any host-side change.
 * Source: brotensor ops/flash_attention.h, flash_attention_decode_len (the
 * valid length is read on the device; query row q of an L_q block sits at
 * position valid_len - L_q + q and attends [0, p]).
 *   lengths : device array of B int32, 4-byte aligned; sequence b holds
 *             L_b = min(max(lengths[b], 0), Tk) valid keys (rows 0 .. L_b-1 of
 *             its cache); keys from L_b on are not visible.  Its Lq query rows
 *             sit at positions L_b - Lq .. L_b - 1 (no q_offset argument);
 *             with causal masking a row at a negative position sees no key
 *             (O = 0, LSE = -inf), as does every row of a sequence with L_b = 0.
 *   Tk      : the cache capacity (rows allocated per sequence); the split plan
 *             and the workspace size depend on it alone.
 *   dt      : ATTN_BF16 or ATTN_F16 (ATTN_F32 returns ATTN_ERR_UNSUPPORTED).
 *   The rest, key_mask included, as for attn_decode.
 */
ATTN_API attn_status attn_decode_len(attn_dtype dt, const void* q, const void* k, const void* v, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, int B, int Lq,
                        int Tk, int H, int Hkv, int hd, float scale, int causal, int window,
                        float softcap, const int* lengths, const float* key_mask,
                        long long key_mask_bstride, void* stream);

/*
 * Forward and backward with a general two-sided window and an additive score
 * bias.
 * Source: ferrotensor engine/attention.rs (flash_attention_v2_with: additive mask
 * [batch, heads, seq_q, seq_k], size-1 dimensions broadcast with stride 0 by
 * mask_strides; AttentionOptions window |p - j| < window), brotensor
 * ops/flash_attention.h, flash_attention_windowed_forward (bidirectional window:
 * keys [p - window/2, p + window/2]) and forge attention.metal, attention_fwd_f32
 * (one-sided window: keys from i + 1 - window on).
 *   window_left, window_right : the query at absolute position p = i + q_offset
 *                sees keys j with p - window_left <= j <= p + window_right; a
 *                negative side is unbounded.  causal = (-1, 0); ferrotensor's
 *                window w = (w-1, w-1), with causal (w-1, 0); brotensor's
 *                bidirectional window w = (w/2, w/2); forge's one-sided window w =
 *                (w-1, -1).
 *   bias       : fp32 added to the (capped) scaled score of (b, h, i, j):
 *                bias[b*bias_sb + h*bias_sh + i*bias_sq + j*bias_sk], strides in
 *                elements (0 broadcasts a dimension), 4-byte aligned; NULL for none.
 *                A -inf entry drops that pair.  The gradient treats it as a constant.
 *   Everything else as attn_fwd / attn_bwd (key mask included).  With a bias,
 *   16-bit calls at hd 64 and 128 run on the tensor cores (with or without a
 *   softcap); at hd 32, 96 and 256 on the CUDA-core kernels (same results, slower).
 */
ATTN_API attn_status attn_fwd_ex(attn_dtype dt, const void* q, const void* k, const void* v, void* o,
                        float* lse, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale,
                        int window_left, int window_right, float softcap, int q_offset,
                        const float* key_mask, long long key_mask_bstride, const float* bias,
                        long long bias_sb, long long bias_sh, long long bias_sq, long long bias_sk,
                        void* stream);

ATTN_API attn_status attn_bwd_ex(attn_dtype dt, const void* q, const void* k, const void* v,
                        const void* o, const void* dout, const float* lse, void* dq, void* dk,
                        void* dv, void* workspace, size_t workspace_bytes, int B, int Tq, int Tk,
                        int H, int Hkv, int hd, float scale, int window_left, int window_right,
                        float softcap, int q_offset, const float* key_mask,
                        long long key_mask_bstride, const float* bias, long long bias_sb,
                        long long bias_sh, long long bias_sq, long long bias_sk, void* stream);

/*
 * Packed variable-length attention: the batch's sequences stored back to back
 * in one tensor, no padding, no attention across sequences.
 * Source: brotensor ops/flash_attention.h, flash_attention_varlen_forward and
 * flash_attention_varlen_backward (cu_seqlens prefix sums on the device;
 * sequence b covers query rows [cu_q[b], cu_q[b+1]) and key rows
 * [cu_k[b], cu_k[b+1]); causal: key j of the sequence is visible to its query
 * i when j <= i, both counted from the sequence's first row).
 *   q, o          : [total_q, H*hd]; k, v : [total_k, Hkv*hd]; 16-byte aligned.
 *   cu_seqlens_q, cu_seqlens_k : device arrays of batch+1 int32 (4-byte aligned),
 *                   non-decreasing, cu[0] >= 0 and cu[batch] <= total.
 *   max_seqlen_q, max_seqlen_k : bounds on every sequence's query / key count;
 *                   the launch shape depends on them (and on batch) alone, so one
 *                   captured graph serves every packing within the bounds.  A
 *                   sequence above the bound or past total (or a decreasing or
 *                   negative prefix sum) is cut to what fits (or to nothing), so no
 *                   access leaves the buffers, and attn_get_device_status() then
 *                   returns ATTN_ERR_INVALID_ARG.
 *   lse           : [batch, H, max_seqlen_q] fp32 or NULL; entry (b, h, i) for
 *                   i < the length of sequence b.
 *   window, softcap, scale, dt, H, Hkv, hd : as for attn_fwd, applied within each
 *                   sequence (query positions from 0, no q_offset, no key mask).
 *   Rows of o outside every sequence are not written.
 */
ATTN_API attn_status attn_varlen_fwd(attn_dtype dt, const void* q, const void* k, const void* v, void* o,
                        float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int H,
                        int Hkv, int hd, float scale, int causal, int window, float softcap,
                        void* stream);

/*
 * Backward of attn_varlen_fwd (same arguments; o and lse from that call).
 * Source: brotensor ops/flash_attention.h, flash_attention_varlen_backward
 * (per-sequence recompute, gradients overwritten).
 * dq [total_q, H*hd], dk and dv [total_k, Hkv*hd] are overwritten on the rows
 * of every sequence (zero where nothing is visible); rows outside every
 * sequence are not written.  workspace: at least
 * attn_bwd_workspace_size(batch, max_seqlen_q, H) bytes, 16-byte aligned.
 */
ATTN_API attn_status attn_varlen_bwd(attn_dtype dt, const void* q, const void* k, const void* v,
                        const void* o, const void* dout, const float* lse, void* dq, void* dk,
                        void* dv, void* workspace, size_t workspace_bytes,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int H,
                        int Hkv, int hd, float scale, int causal, int window, float softcap,
                        void* stream);

/*
 * Packed bidirectional self-attention straight off a fused QKV projection.
 * Source: brotensor ops/flash_attention.h, flash_attention_packed_qkv_forward /
 * flash_attention_packed_qkv_backward (many sequences of any lengths packed back to
 * back in one row block, rows attending only inside their own sequence, an optional
 * bidirectional window; the backward recomputes the softmax from q, k and v).
 *   qkv        : [L][3*H*hd], each row [q heads | k heads | v heads], 16-byte aligned.
 *   seq_bounds : [L][2] int32 on the device, 8-byte aligned: row r's sequence is rows
 *                [seq_bounds[r][0], seq_bounds[r][1]), a range holding r; sequences
 *                lie back to back, so the bounds never decrease down the rows (the
 *                kernels rely on it to pick each tile's keys; bounds past [0, L) are
 *                clipped).  Membership is data: the launch shape depends on L only.
 *   window     : >= 0; > 0: row r sees keys j of its sequence with |r - j| <= window/2
 *                (integer division); 0: every key of its sequence.  Non-causal.
 *   scale      : > 0 (1/sqrt(hd) in the usual case).  H: heads (no grouping).
 *   attn_packed_qkv_fwd : o [L][H*hd] (overwritten); lse [H][L] fp32, or NULL.
 *   attn_packed_qkv_bwd : dqkv [L][3*H*hd] (overwritten), each row [dq | dk | dv], from
 *                dout [L][H*hd]; O and LSE are formed again from qkv.
 *   workspace  : at least attn_packed_qkv_workspace_size(dt, L, H, hd, backward) bytes,
 *                16-byte aligned; contents on entry are ignored.  16-bit rows at hd
 *                64 / 128 run on the tensor cores, whose tensor maps read q, k and v
 *                in place from the rows (and the backward writes dq, dk, dv straight
 *                into the dqkv rows); the workspace then holds only the order in which
 *                the row blocks run (heaviest first, formed on the stream by a small
 *                kernel from seq_bounds) and the backward's O, LSE and D.  Other types
 *                and head sizes run on the CUDA-core kernels
 *                over contiguous copies of q, k and v made in the workspace (strided
 *                copies on the stream), the backward's gradients copied into dqkv.
 *   Errors as attn_fwd; L = 0 is a no-op.
 */
ATTN_API size_t attn_packed_qkv_workspace_size(attn_dtype dt, int L, int H, int hd, int backward);
ATTN_API attn_status attn_packed_qkv_fwd(attn_dtype dt, const void* qkv, const int* seq_bounds, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, int L, int H, int hd,
                        float scale, int window, void* stream);
ATTN_API attn_status attn_packed_qkv_bwd(attn_dtype dt, const void* qkv, const void* dout,
                        const int* seq_bounds, void* dqkv, void* workspace, size_t workspace_bytes,
                        int L, int H, int hd, float scale, int window, void* stream);

/*
 * attn_decode without a workspace argument, for callers that cannot call
 * cudaMalloc and have no scratch buffer to pass in: for example a plugin that
 * is handed only its input and output buffers, a serving loop that forbids
 * device allocation after start-up so that a request can never fail for lack
 * of memory, or a C caller with no device allocator of its own.  None of the
 * sources cited in this header defines such a call; it exists for those callers.
 *
 * Same arguments, kernels and results as attn_decode.  The split partials
 * live in one fixed array of 32 MiB that the library reserves in device
 * memory on every GPU that loads it, held until the process exits; shapes
 * whose attn_decode_workspace_size() exceeds 32 MiB return
 * ATTN_ERR_UNSUPPORTED and launch nothing.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 * The first call on a device looks up the array's device address (a one-time
 * set-up step), so make that first call before any stream capture.  All calls
 * share the one array and it keeps the last call's contents (no entry needs to
 * start at zero: each call writes every partial it later reads); calls that
 * overlap on the GPU, for example on two streams, race on it.
 */
ATTN_API attn_status attn_decode_noalloc(attn_dtype dt, const void* q, const void* k, const void* v,
                        void* o, float* lse, int B, int Lq, int Tk, int H, int Hkv, int hd,
                        float scale, int causal, int window, float softcap, int q_offset,
                        const float* key_mask, long long key_mask_bstride, void* stream);

/*
 * Rotate-half rotary embedding, in place, for the q or k given to the calls
 * above (a separate HBM-bound pass: the attention kernels read the rotated rows).
 * Source: ferrotensor engine/attention.rs, rope / rope_theta (the rotate-half
 * form, done in place, with base 10000 unless set; every head vector of token s
 * gets position pos + s).
 *   x     : [B, T, H*hd] of dtype dt, 16-byte aligned; overwritten.
 *   pos   : position of token 0 of every sequence (>= 0).
 *   theta : base frequency (10000 in the page's default, > 0).
 *   Pair (x[i], x[i + hd/2]) of each head vector, i < hd/2, turns by
 *   (pos + s) * theta^(-2i/hd).  hd a multiple of 4 in [4, 256].
 */
ATTN_API attn_status attn_rope(attn_dtype dt, void* x, int B, int T, int H, int hd, int pos, float theta,
                        void* stream);

/*
 * Attention on rotary-embedded queries and keys, for callers that keep q and k
 * unrotated.  Source: ferrotensor engine/attention.rs, rope / rope_theta (the
 * rotate-half turn applied to q and k before flash attention), with the turn of
 * attn_rope: pair (x[c], x[c + hd/2]) of a head vector at rotary position t turns
 * by t * rope_theta^(-2c/hd).  Query row i sits at rotary position
 * rope_pos + q_offset + i and key j at rope_pos + j, the positions the causal and
 * window rules use, shifted by rope_pos >= 0.
 *   attn_fwd_rope : O and LSE of attention on the turned q and k; q and k are not
 *                   modified.  16-bit hd 64 / 128 turn the query tiles inside the
 *                   forward kernel (from a cosine/sine table in the workspace);
 *                   the keys are turned into the workspace first (one pass over k).
 *                   Other types and head sizes turn q into the workspace too.  The
 *                   result equals attn_rope on q and k followed by attn_fwd, bit for
 *                   bit.  workspace: at least attn_fwd_rope_workspace_size() bytes,
 *                   16-byte aligned; contents on entry are ignored.
 *   attn_bwd_rope : the gradients of the unrotated q and k (dq = R^T dq', dk =
 *                   R^T dk' for the turned operands' gradients dq', dk') and dv,
 *                   overwritten; o and lse come from attn_fwd_rope with the same
 *                   arguments.  It turns q and k into the workspace, runs the
 *                   backward on them and turns dq and dk back in place.  workspace:
 *                   at least attn_bwd_rope_workspace_size() bytes, 16-byte aligned.
 *   rope_theta > 0 and finite; hd a multiple of 4.  The rest as attn_fwd / attn_bwd.
 */
ATTN_API size_t attn_fwd_rope_workspace_size(attn_dtype dt, int B, int Tq, int Tk, int H, int Hkv, int hd,
                        int q_offset);
ATTN_API attn_status attn_fwd_rope(attn_dtype dt, const void* q, const void* k, const void* v, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, int B, int Tq, int Tk, int H,
                        int Hkv, int hd, float scale, int causal, int window, float softcap, int q_offset,
                        const float* key_mask, long long key_mask_bstride, int rope_pos, float rope_theta,
                        void* stream);
ATTN_API size_t attn_bwd_rope_workspace_size(attn_dtype dt, int B, int Tq, int Tk, int H, int Hkv, int hd);
ATTN_API attn_status attn_bwd_rope(attn_dtype dt, const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                        size_t workspace_bytes, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale,
                        int causal, int window, float softcap, int q_offset, const float* key_mask,
                        long long key_mask_bstride, int rope_pos, float rope_theta, void* stream);

/* Human-readable name of a status code (static storage). */
ATTN_API const char* attn_status_string(attn_status s);

/*
 * Reads and clears the device status word that bounded waits set when they
 * run out (and that packed-sequence calls set when cu_seqlens break their
 * bounds).  Synchronises `stream` first.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a
 * wait ran out), ATTN_ERR_INVALID_ARG (only the cu_seqlens bit is set) or
 * ATTN_ERR_CUDA.  If `detail` is not NULL it receives the raw word (which wait
 * gave up, as a bit set; bit 9: cu_seqlens out of bounds).
 */
ATTN_API attn_status attn_get_device_status(void* stream, unsigned int* detail);

/*
 * Self-test of the bounded-wait path: launches one CTA that waits on a
 * barrier nothing will complete, for at most `timeout_us` microseconds
 * (1 .. 2000000), then sets the status word and exits normally.  The caller
 * then sees ATTN_ERR_TIMEOUT from attn_get_device_status().
 */
ATTN_API attn_status attn_selftest_bounded_wait(unsigned int timeout_us, void* stream);

/* Which kernel family attn_fwd (and attn_fwd_ex without a bias) uses for (dt, hd):
 * 0 = CUDA-core kernels, 1 = tcgen05 tensor cores.  16-bit hd 32, 64, 96, 128 and 256
 * run on the tensor cores. */
ATTN_API int attn_kernel_family(attn_dtype dt, int hd);

/* The same for attn_bwd (without a bias): 16-bit hd 32, 64, 96, 128 and 256 run on
 * the tensor cores. */
ATTN_API int attn_kernel_family_bwd(attn_dtype dt, int hd);

/* Running total of kernels this library has enqueued in this process. */
ATTN_API unsigned long long attn_launch_count(void);

/* ABI version, bumped on any signature change. */
ATTN_API int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
