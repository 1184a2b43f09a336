/*
 * k6attn.h -- C ABI of libk6attn: joint-sequence attention for long-context
 * video diffusion transformers on one NVIDIA GB300 (sm_103a).
 *
 * The path: rotary embeddings on Q and K, full non-causal multi-head attention
 * over the joint sequence (video tokens followed by text/audio tokens),
 * computed per K/V chunk with online softmax into partial outputs and their
 * log-sum-exp, the log-sum-exp merge of those partials, and the
 * sequence-partitioned <-> head-partitioned relayout.
 *
 * Sources (web pages; section names in quotes):
 *  [USP]  xDiT PR #586 "KV-cache and joint tensors for USP": "How?" (joint
 *         tensors), the USP dispatch listing (`_attention`, `ring_attn`,
 *         `_ft_c_input_all_to_all`, `_ft_c_output_all_to_all`).
 *  [CP]   "Context Parallelism in vLLM Omni Neuron": "Ring attention (current
 *         implementation)", "Self-Attention with Context Parallelism",
 *         "Comparison with Other CP Strategies", "Positional Embedding
 *         Handling", "Scaling Properties", "Sequence Length Constraints".
 *  [K6]   vLLM-Omni recipe "Kandinsky 6 TI2VA -- H100", section "Notes", its
 *         sequence-parallel item: the visual tokens and their rotary tables are
 *         split across ranks, and the audio queries attend over every visual
 *         token.
 *
 * Conventions shared by every call:
 *  - Tensors are caller-owned DEVICE pointers, 16-byte aligned, densely packed
 *    in the stated layout.  The library never allocates or frees them.
 *  - Layout BSHD: q [B][Sq][H][d] with Sq = Nv + Nj, video rows first and the
 *    Nj joint rows at the rear; k, v [B][Nv][H][d]; joint_k, joint_v
 *    [B][Nj][H][d].  The key/value sequence is concat(k, joint_k) along the
 *    token axis (length Sk = Nv + Nj = Sq).
 *  - Element type: K6ATTN_BF16 (storage bf16, products fp32-accumulated,
 *    softmax fp32) or K6ATTN_F32 (everything fp32, no tf32).
 *  - lse arrays are fp32 [B][H][Sq], natural log of sum_j exp(s_ij) with
 *    s_ij = q~_i . k~_j / sqrt(d).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream and returns after enqueueing.
 *  - A handle belongs to the device that was current at k6attn_create (its
 *    rotary tables and error word live there).  Every call that takes a handle,
 *    except k6attn_destroy and the host-only queries, must be made with that
 *    device current; otherwise it returns K6ATTN_ERR_INVALID_ARG and launches
 *    nothing.
 *  - Calls never abort or trap.  Argument errors are found on the host before
 *    any launch and return K6ATTN_ERR_INVALID_ARG / _UNSUPPORTED /
 *    _WORKSPACE; k6attn_last_error() then holds a message (thread-local).
 *    Device-side waits are bounded; a wait that runs out sets the handle's
 *    device error word, which k6attn_sync() reports as K6ATTN_ERR_TIMEOUT.
 */
#ifndef K6ATTN_H
#define K6ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    K6ATTN_OK = 0,
    K6ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, indivisible split, aliasing, misalignment */
    K6ATTN_ERR_UNSUPPORTED = 2, /* valid request the library does not implement (e.g. bf16 with d != 128) */
    K6ATTN_ERR_CUDA = 3,        /* a CUDA runtime call failed; message in k6attn_last_error() */
    K6ATTN_ERR_TIMEOUT = 4,     /* a device-side wait ran out (reported by k6attn_sync) */
    K6ATTN_ERR_WORKSPACE = 5,   /* workspace pointer null or smaller than k6attn_workspace_bytes() */
    K6ATTN_ERR_RANGE = 6        /* a rotated q/k value is not finite in fp16 (reported by k6attn_sync) */
} k6attn_status;

/* Storage types.  A handle's dtype (BF16 or F32) is the type of q, k, v,
 * joint_k, joint_v and out.  F16 is only a type for ROTATED q/k/joint_k of a
 * BF16 handle: rounding the rotated values to fp16 (11-bit significand)
 * instead of bf16 (8-bit) cuts the error they add to the logits 8-fold, at the
 * same tensor-core rate (Q.K^T runs fp16 x fp16, P.V bf16 x bf16, both with
 * fp32 accumulation).  E4M3 (8-bit float, 3 mantissa bits, finite range
 * +-448) is likewise only a type for rotated q/k/joint_k of a BF16 handle: the
 * FP8 mode, where Q.K^T runs on e4m3 operands (kind::f8f6f4, half the tensor
 * instructions of 16-bit operands) and P.V stays bf16; its error is that of
 * rounding q and k to 3 mantissa bits (2^-4 relative), 16 times fp16's. */
typedef enum { K6ATTN_BF16 = 0, K6ATTN_F32 = 1, K6ATTN_F16 = 2, K6ATTN_E4M3 = 3 } k6attn_dtype;

/*
 * Problem descriptor, fixed at handle creation.
 *  B, H, d       batch, heads, head dim.  d in {64, 128} for F32; d == 128 for BF16.
 *  grid_t/h/w    video latent grid; Nv = grid_t * grid_h * grid_w video tokens,
 *                flattened row-major (t slowest, w fastest).
 *  axis_dim[3]   head dims owned by the t, h, w rotary axes, in that order,
 *                each even, summing to d (e.g. 32,48,48 for d = 128; 0,64,64
 *                for 2-D image grids).
 *  theta         rotary base (10000).
 *  n_joint       Nj joint (text/audio) tokens, appended after the video tokens
 *                on both the query and the key/value side ([USP] "How?").
 *  joint_rope    0: joint tokens are not rotated; 1: joint token j turns by a
 *                1-D rotary over the full head dim at position j.
 * Rotary reading (the pages print no formula; [CP] "Positional Embedding
 * Handling" shows per-token cos/sin tables): pair i of an axis segment, dims
 * (2i, 2i+1) of that segment, turns by pos * theta^(-2i/d_axis) as a complex
 * product.
 */
typedef struct {
    int B, H, d;
    k6attn_dtype dtype;
    int grid_t, grid_h, grid_w;
    int axis_dim[3];
    double theta;
    int n_joint;
    int joint_rope;
} k6attn_desc;

typedef struct k6attn_handle *k6attn_t;

/* Validate `desc`, build the per-axis rotary tables on the current device and
 * allocate the handle's device error word.  On success *out owns them. */
k6attn_status k6attn_create(const k6attn_desc *desc, k6attn_t *out);

/* Free the handle and what it owns (synchronises the device first).  NULL is a no-op. */
void k6attn_destroy(k6attn_t h);

/* Device pointer and byte size of the handle-owned rotary tables (fp32 cos/sin
 * pairs: axis t [grid_t][axis_dim0/2], axis h [grid_h][axis_dim1/2], axis w
 * [grid_w][axis_dim2/2], then, when joint_rope == 1, joint [Nj][d/2]).
 * Pass this pointer as `rope_tables` below. */
const void *k6attn_rope_tables(k6attn_t h);
size_t k6attn_rope_tables_bytes(k6attn_t h);

/* Workspace bytes k6attn_forward needs for `n_chunks` K/V chunks, with
 * (with_rope = 1) or without the rotated copies of q/k/joint_k:
 *   rotated copies  (B*Sq*H*d + B*Nv*H*d + B*Nj*H*d) * elem   if with_rope
 *   partial outputs n * B*Sq*H*d * 4 + n * B*H*Sq * 4          if n_chunks > 1
 *   (room for one partial per chunk; with chunk groups only the first
 *   n_chunks / k6attn_chunk_group(h, n_chunks) are written)
 * (each region rounded up to 256 bytes).  0 when neither applies. */
size_t k6attn_workspace_bytes(k6attn_t h, int n_chunks, int with_rope);

/*
 * Rotary embedding of q, k and joint_k, one fused launch ([CP]
 * "Self-Attention with Context Parallelism": `apply_rotary_emb_wan` on query
 * and key; [K6] RoPE travels with the visual tokens).
 *  q        [B][Sq][H][d]; row n < Nv at its video grid position, row n >= Nv
 *           is joint token n - Nv.
 *  k        [B][Nv][H][d] video keys.
 *  joint_k  [B][Nj][H][d] (may be NULL when Nj == 0).
 *  rope_tables  k6attn_rope_tables(h) or a caller copy in the same layout.
 *  q_out, k_out, joint_k_out  destinations in the same layouts, of type
 *           out_dtype.  Equal to the sources for in-place rotation (then
 *           out_dtype must be the handle's dtype); otherwise disjoint from
 *           every source.  out_dtype F16 is allowed for BF16 handles.
 * Rotation in fp32, rounded to nearest even.  Writing F16, a value that is
 * not finite in fp16 sets the handle's error word (K6ATTN_ERR_RANGE at
 * k6attn_sync).
 */
k6attn_status k6attn_rope_qk(k6attn_t h, const void *q, const void *k, const void *joint_k, const void *rope_tables,
                             void *q_out, void *k_out, void *joint_k_out, k6attn_dtype out_dtype, void *stream);

/*
 * QK-norm, then rotary embedding, in one launch ([CP] "Self-Attention with
 * Context Parallelism": `norm_q(q)` / `norm_k(k)` on the projected rows, then
 * `apply_rotary_emb_wan`; "Distributed Normalization": the RMS statistic is
 * taken over the hidden dim).  Each token row of H*d values is RMS-normalised
 * in fp32 as y = x / sqrt(mean(x^2) + eps) * w, then rotated exactly as
 * k6attn_rope_qk does; arguments and outputs as there, plus:
 *  q_weight, k_weight   fp32 [H*d] device arrays for video query / key rows.
 *  joint_q_weight, joint_k_weight  fp32 [H*d] for the joint query rows (the
 *           rear Nj rows of q) and for joint_k; NULL = use q_weight/k_weight.
 *  eps      >= 0.
 * The norm needs each token's full row, so call it on sequence-partitioned
 * (full-head) tensors, before a seq->head relayout.
 */
k6attn_status k6attn_norm_rope_qk(k6attn_t h, const void *q, const void *k, const void *joint_k,
                                  const float *q_weight, const float *k_weight, const float *joint_q_weight,
                                  const float *joint_k_weight, float eps, const void *rope_tables, void *q_out,
                                  void *k_out, void *joint_k_out, k6attn_dtype out_dtype, void *stream);

/*
 * Joint-sequence attention forward ([USP] `_attention`; [CP] "Ring attention
 * (current implementation)": each K/V chunk is attended separately and the
 * partials combine through their log-sum-exp).
 *  q, k, v, joint_k, joint_v  inputs in the layouts above (joint_* may be NULL
 *           when Nj == 0).  Not modified.
 *  rope_tables  NULL: q/k/joint_k are already rotated (handle dtype).
 *           Otherwise rotated copies are written to the workspace first
 *           (k6attn_rope_qk math; fp16 copies for a BF16 handle, so a
 *           rotated value must be finite in fp16: K6ATTN_ERR_RANGE at
 *           k6attn_sync otherwise; bf16 copies with K6ATTN_OPT_ROTATE_BF16).
 *  n_chunks K/V chunks: chunk c covers keys [c*Sk/n, (c+1)*Sk/n) of
 *           concat(k, joint_k); Sk % n_chunks must be 0 ([CP] "Sequence
 *           Length Constraints").  n_chunks == 1 writes out/lse directly;
 *           otherwise the chunks run in groups of k6attn_chunk_group(h,
 *           n_chunks), each merged inside the kernel, and the n_chunks / group
 *           fp32 partials (workspace) are merged by the k6attn_lse_merge
 *           kernel (none when n_chunks / group == 1).
 *  out      [B][Sq][H][d], same element type as q.  Must not alias any input.
 *  lse      fp32 [B][H][Sq] (may be NULL: not written).
 *  workspace, workspace_bytes  caller-owned device scratch of at least
 *           k6attn_workspace_bytes(h, n_chunks, rope_tables != NULL); may be
 *           NULL when that is 0.
 */
k6attn_status k6attn_forward(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                             const void *joint_v, const void *rope_tables, int n_chunks, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * The attention step alone, on already-rotated inputs: for each K/V chunk c
 * (as in k6attn_forward) the chunk's softmax(q k^T / sqrt(d)) v and its
 * log-sum-exp ([CP] "Ring attention (current implementation)").
 *  n_chunks == 1: out is [B][Sq][H][d] in the handle's element type and lse
 *           fp32 [B][H][Sq] (may be NULL).
 *  n_chunks > 1:  out is fp32 partials [n_chunks][B][Sq][H][d] and lse fp32
 *           [n_chunks][B][H][Sq] (required); combine them with
 *           k6attn_lse_merge.
 *  qk_dtype the type of q, k and joint_k: the handle's dtype, or F16 for a
 *           BF16 handle (v and joint_v always have the handle's dtype), or
 *           E4M3 for a BF16 handle: Q.K^T then runs on 8-bit operands, P.V
 *           as before.
 * Inputs as in k6attn_forward; outputs must not alias them.
 */
k6attn_status k6attn_attention_chunks(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                                      const void *joint_v, k6attn_dtype qk_dtype, int n_chunks, void *out, float *lse,
                                      void *stream);

/*
 * Chunk groups: the attention step over n_chunks K/V chunks in which each
 * group of `group` consecutive chunks (group divides n_chunks) is merged
 * inside the kernel, so that it leaves n_chunks / group partials instead of
 * n_chunks ([CP] "Ring attention (current implementation)": the chunks'
 * partials combine through their log-sum-exp, and that combine is
 * associative).  Within a group the merge happens in tensor memory: the row
 * maximum, row sum and unnormalised output of the chunks so far carry into the
 * next chunk, whose tiles rescale them exactly as the tiles of one chunk do;
 * the groups are then combined by k6attn_lse_merge / k6attn_lse_merge_heads.
 *  group == 1 is k6attn_attention_chunks.  group > 1 needs a BF16 handle.
 *  n_chunks / group == 1: out is [B][Sq][H][d] (handle type) and lse fp32
 *           [B][H][Sq] (may be NULL) -- the attention of the whole sequence.
 *  n_chunks / group > 1: out is fp32 [n_chunks/group][B][Sq][H][d], lse fp32
 *           [n_chunks/group][B][H][Sq] (required); partial g covers chunks
 *           [g*group, (g+1)*group).
 * Other arguments as in k6attn_attention_chunks.
 *
 * k6attn_chunk_group: the group the library itself uses for n_chunks chunks of
 * this handle's problem on the current device (k6attn_forward and
 * k6attn_cross_forward use it): the largest divisor of n_chunks up to 4 that
 * still leaves at least four waves of CTAs, 1 for F32 handles; 0 for a null
 * handle or n_chunks < 1.
 */
int k6attn_chunk_group(k6attn_t h, int n_chunks);
k6attn_status k6attn_attention_chunk_groups(k6attn_t h, const void *q, const void *k, const void *v,
                                            const void *joint_k, const void *joint_v, k6attn_dtype qk_dtype,
                                            int n_chunks, int group, void *out, float *lse, void *stream);

/*
 * The Ulysses prologue of one attention layer, one pass over HBM: rotary
 * embeddings of q, k and joint_k (as k6attn_rope_qk) and the
 * sequence->head relayout of q, k, joint_k, v and joint_v ([CP]
 * "Self-Attention with Context Parallelism": rotary on the local tokens before
 * attention; [USP] `_ft_c_input_all_to_all`; [CP] "Comparison with Other CP
 * Strategies").  BF16 handles (d = 128); h describes the full problem
 * (B, H heads).  P divides H; with Hl = H / P, for each tensor x of R rows
 * per batch (R = Sq for q, Nv for k and v, Nj for joint_k and joint_v):
 *   x_out[p][b][n][hh][e] = rot(x[b][n][p*Hl + hh][e])   (q, k, joint_k)
 *   x_out[p][b][n][hh][e] =     x[b][n][p*Hl + hh][e]    (v, joint_v, bit copy)
 * i.e. each output is [P][B][R][Hl][d]: the input of a handle with batch P*B
 * and Hl heads.  For B == 1 this equals k6attn_rope_qk into copies followed by
 * k6attn_seq2head_relayout of each tensor (bit for bit).
 *  qk_out_dtype  BF16, F16 or E4M3: the type of q_out, k_out, joint_k_out
 *           (v_out and joint_v_out are bf16).  F16: a rotated value that is
 *           not finite in fp16 sets K6ATTN_ERR_RANGE (at k6attn_sync); E4M3: a
 *           rotated value beyond +-448 is stored as +-448 and sets it too.
 *  joint_* may be NULL when Nj == 0.  Outputs must not overlap any input or
 *  one another.
 */
k6attn_status k6attn_rope_split_heads(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                                      const void *joint_v, const void *rope_tables, int P, k6attn_dtype qk_out_dtype,
                                      void *q_out, void *k_out, void *v_out, void *joint_k_out, void *joint_v_out,
                                      void *stream);

/*
 * The Ulysses epilogue: the log-sum-exp merge of partials computed on the
 * head-partitioned layout, written straight to the sequence layout ([CP]
 * "Ring attention (current implementation)"; [USP]
 * `_ft_c_output_all_to_all`).  h describes the full problem (B, H heads);
 * P divides H and Hl = H / P.
 *  part_o   fp32 [n_parts][P*B][Sq][Hl][d], part_lse fp32 [n_parts][P*B][Hl][Sq]:
 *           partials of the handle with batch P*B and Hl heads (as written by
 *           k6attn_attention_chunks or k6attn_attention_chunk_groups on
 *           inputs from k6attn_rope_split_heads).
 *  out      [B][Sq][H][d] in the handle's type, lse fp32 [B][H][Sq] (may be
 *           NULL): head p*Hl + hh of batch b holds the merge of problem
 *           p*B + b, head hh.  P == 1 is k6attn_lse_merge.
 */
k6attn_status k6attn_lse_merge_heads(k6attn_t h, const float *part_o, const float *part_lse, int n_parts, int P,
                                     void *out, float *lse, void *stream);

/*
 * Backward pass of the joint attention (the pages describe inference only;
 * these are the chain-rule gradients of out = softmax(s) v with
 * s = q k^T / sqrt(d), over concat(k, joint_k) as in k6attn_attention_chunks
 * with one chunk):
 *   D_i = sum_e dout_ie out_ie,  P = exp(s - lse),
 *   dS  = P o (dout v^T - D),    dv = P^T dout,
 *   dq  = dS k / sqrt(d),        dk = dS^T q / sqrt(d).
 * The q/k gradients are with respect to the q, k given (the rotated copies
 * when rotary embeddings are used).  BF16 handles with d = 128.
 *  q, k, joint_k  rotated inputs, type qk_dtype (BF16 or F16); v, joint_v
 *           bf16; layouts as above.  Not modified.
 *  out, lse the forward result for these inputs (out bf16 [B][Sq][H][d], lse
 *           fp32 [B][H][Sq], as written by k6attn_attention_chunks with one
 *           chunk or by k6attn_forward).
 *  dout     bf16 [B][Sq][H][d], the gradient of the loss with respect to out.
 *  dq       fp32 [B][Sq][H][d]; dk, dv fp32 [B][Nv][H][d]; djoint_k,
 *           djoint_v fp32 [B][Nj][H][d] (may be NULL when Nj == 0).  Fully
 *           overwritten; must not alias any input or one another.
 *  workspace, workspace_bytes  caller-owned device scratch of at least
 *           k6attn_backward_workspace_bytes(h) bytes (per (b, h, row) the
 *           row's lse in base 2 and D_i, 8 bytes).
 * P is rounded to bf16 and dS to qk_dtype before their products; all
 * products accumulate in fp32.
 */
size_t k6attn_backward_workspace_bytes(k6attn_t h);
k6attn_status k6attn_backward(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                              const void *joint_v, k6attn_dtype qk_dtype, const void *out, const void *dout,
                              const float *lse, float *dq, float *dk, float *dv, float *djoint_k, float *djoint_v,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Constant-max softmax ([CP] "Related information": the ring kernel
 * `ring_attention_const_max_fwd` uses a runtime bound on the softmax maximum
 * instead of a running maximum, so no partial output is ever rescaled).  The
 * pages do not give the bound; this library uses Cauchy-Schwarz:
 *   bound_i = |q_i| * max_j |k_j| / sqrt(d)  >=  every logit of row i,
 * the maximum taken over all keys of the (batch, head) pair, so one bound
 * serves every K/V chunk and the partials merge unchanged.
 *
 * k6attn_row_bounds: bounds fp32 of k6attn_row_bounds_bytes(h) bytes: the
 *   first B*H*Sq floats are the row bounds [B][H][Sq] (natural-log units of
 *   the logits), the last B*H the key-norm maxima.  q/k/joint_k as for
 *   k6attn_attention_chunks (rotated; qk_dtype the handle's or F16).
 * k6attn_attention_chunks_bounded: k6attn_attention_chunks with the bounds
 *   in place of the running maximum (bf16 handles).  Exactly the same
 *   mathematics; a row whose every term underflows (a bound more than about
 *   87 above its largest logit) sets the error word (K6ATTN_ERR_RANGE at
 *   k6attn_sync) and gets a zero output.
 * k6attn_attention_chunk_groups_bounded: the same with each CTA's group of
 *   `group` consecutive chunks merged in the kernel (as
 *   k6attn_attention_chunk_groups): n_chunks / group partials, or out/lse
 *   directly when that is 1.  With one bound for every chunk, the merge inside
 *   a group is a plain sum of the chunks' terms.
 */
size_t k6attn_row_bounds_bytes(k6attn_t h);
k6attn_status k6attn_row_bounds(k6attn_t h, const void *q, const void *k, const void *joint_k, k6attn_dtype qk_dtype,
                                float *bounds, void *stream);
k6attn_status k6attn_attention_chunks_bounded(k6attn_t h, const void *q, const void *k, const void *v,
                                              const void *joint_k, const void *joint_v, k6attn_dtype qk_dtype,
                                              const float *bounds, int n_chunks, void *out, float *lse,
                                              void *stream);
k6attn_status k6attn_attention_chunk_groups_bounded(k6attn_t h, const void *q, const void *k, const void *v,
                                                    const void *joint_k, const void *joint_v, k6attn_dtype qk_dtype,
                                                    const float *bounds, int n_chunks, int group, void *out,
                                                    float *lse, void *stream);

/*
 * Log-sum-exp merge of per-chunk partials (ring attention's combine step,
 * [CP] "Ring attention (current implementation)", "Scaling Properties"):
 *   LSE = log sum_c exp(LSE_c),  out = sum_c exp(LSE_c - LSE) * O_c.
 *  part_o   fp32 [n_chunks][B][Sq][H][d];  part_lse fp32 [n_chunks][B][H][Sq].
 *  out      [B][Sq][H][d] in the handle's element type;  lse fp32 [B][H][Sq]
 *           (may be NULL).  Outputs must not alias the partials.
 */
k6attn_status k6attn_lse_merge(k6attn_t h, const float *part_o, const float *part_lse, int n_chunks, void *out,
                               float *lse, void *stream);

/*
 * Cross-attention: Sq query rows of one stream over Sk keys/values of another
 * ([K6] "Notes", sequence-parallel item: audio queries attend over every
 * visual token; [CP] "Forward Pass Flow": cross-attention reads the encoder
 * states unsharded).  No rotary, no joint
 * tokens; the handle supplies B, H, d, the element type and the error word
 * (its video grid and joint settings are not used).
 *  q        [B][Sq][H][d];  k, v [B][Sk][H][d]  (handle dtype).
 *  n_chunks K/V chunks of Sk/n_chunks keys each (Sk % n_chunks == 0),
 *           combined by their log-sum-exp as in k6attn_forward.
 *  out      [B][Sq][H][d];  lse fp32 [B][H][Sq] (may be NULL).
 *  workspace  at least k6attn_cross_workspace_bytes(h, Sq, n_chunks) bytes;
 *           NULL is accepted when n_chunks == 1.
 * The merged result does not depend on how the keys are split, so the call
 * may run the chunks in finer pieces: for Sq <= 128 (BF16) each chunk may be
 * split into up to 4 sub-chunks, so that the few, HBM-bound CTAs fill the
 * GPU's last wave.  k6attn_cross_workspace_bytes allows for that; with a
 * smaller workspace (or none, for one chunk) the chunks run unsplit.
 */
size_t k6attn_cross_workspace_bytes(k6attn_t h, long Sq, int n_chunks);
k6attn_status k6attn_cross_forward(k6attn_t h, const void *q, long Sq, const void *k, const void *v, long Sk,
                                   int n_chunks, void *out, float *lse, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * Sequence-partitioned <-> head-partitioned relayout, the single-GPU form of
 * the Ulysses all-to-all ([USP] `_ft_c_input_all_to_all` /
 * `_ft_c_output_all_to_all`; [CP] "Comparison with Other CP Strategies").
 * A bit-exact permutation; no arithmetic.  With Sl = S/P and Hl = H/P:
 *   seq  buffer [P][B][Sl][H][d]  (part r holds tokens [r*Sl, (r+1)*Sl))
 *   head buffer [P][B][S][Hl][d]  (part p holds heads  [p*Hl, (p+1)*Hl))
 *   direction 0 (seq -> head): head[p][b][r*Sl+s][hh][e] = seq[r][b][s][p*Hl+hh][e]
 *   direction 1 (head -> seq): the inverse.
 * For B == 1 the seq buffer is byte-identical to a contiguous [1][S][H][d].
 *  elem_bytes 2 or 4.  Requires S % P == 0 and H % P == 0 (INVALID_ARG
 *  otherwise, like [CP]'s ValueError for 3645 tokens on 8 ranks), and
 *  non-overlapping src/dst.  No handle needed.
 */
k6attn_status k6attn_seq2head_relayout(const void *src, void *dst, int B, long S, int H, int d, int elem_bytes,
                                       int P, int direction, void *stream);

/*
 * Forward pass with library-held scratch, for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point; it exists
 * for users of the library, not for the method.
 *
 * Same arguments, computation and results as k6attn_forward without the
 * workspace: the scratch (rotated q/k copies, per-chunk partials) lives in one
 * statically sized device array inside the library, so the call never
 * allocates device memory (no cudaMalloc, no cudaFree, no allocating library
 * routine).  It is meant for code that may not or cannot allocate: a plugin
 * whose host framework owns every device allocation, a deployment held to a
 * memory budget fixed at start-up, a binding that only receives tensors.
 *  - Limit: k6attn_workspace_bytes(h, n_chunks, rope_tables != NULL) must not
 *    exceed K6ATTN_STATIC_SCRATCH_BYTES (32 MiB); a larger problem returns
 *    K6ATTN_ERR_WORKSPACE with a message and launches nothing (use
 *    k6attn_forward with a caller workspace then).
 *  - Every GPU that loads the library reserves the array until the process
 *    exits.
 *  - The first call in a CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress) and keeps it for that context: once per device,
 *    and once more after cudaDeviceReset, which gives the device a new context
 *    with a new copy of the array (the old copy's contents are gone).  Make
 *    that first call, with the handle's device current, before any stream
 *    capture begins.
 *  - All calls on one device share the array, which keeps the last call's
 *    contents: calls that can overlap on the GPU (several streams, or several
 *    host threads without ordering between them) race on it.  Keep such calls
 *    on one stream, or use k6attn_forward.
 *  - Nothing in the array needs to start at zero: a call writes every scratch
 *    byte before reading it.
 */
#define K6ATTN_STATIC_SCRATCH_BYTES (32u << 20)
k6attn_status k6attn_forward_static_scratch(k6attn_t h, const void *q, const void *k, const void *v,
                                            const void *joint_k, const void *joint_v, const void *rope_tables,
                                            int n_chunks, void *out, float *lse, void *stream);

/* Synchronise `stream`, then read and clear the handle's device error word:
 * K6ATTN_ERR_TIMEOUT if any kernel of this handle gave up on a wait,
 * K6ATTN_ERR_RANGE if a rotation into fp16 overflowed or a constant-max row
 * underflowed,
 * K6ATTN_ERR_CUDA on an asynchronous CUDA error, or if the device placed
 * the attention kernel's dynamic shared memory off a 1024-byte boundary (the
 * kernel then computes nothing; its tiles need that alignment and its 227 KB
 * plan leaves no room to realign), else K6ATTN_OK. */
k6attn_status k6attn_sync(k6attn_t h, void *stream);

/* Handle options.
 *  K6ATTN_OPT_WAIT_LIMIT_NS   upper bound, in nanoseconds, on any single
 *      device-side wait of this handle's kernels (default 2e9).  0 makes every
 *      wait give up at once, which tests use to exercise the timeout path
 *      without hanging the GPU.
 *  K6ATTN_OPT_STRICT_MMA_ORDER  accepted (0 or 1) and without effect: the
 *      bf16 kernel always waits for a P.V product to finish reading P before a
 *      Q.K^T product rewrites the tensor memory that holds it, so results do
 *      not depend on the order in which the tensor pipe runs MMAs.
 *  K6ATTN_OPT_ROTATE_BF16  1: k6attn_forward and k6attn_forward_static_scratch
 *      keep the rotated q/k copies of a BF16 handle in bf16, whose range is
 *      that of fp32, instead of fp16 (default 0).  fp16 copies add 8 times less
 *      rounding error to the logits but fail (K6ATTN_ERR_RANGE) on a rotated
 *      value beyond 65,504, which bf16 inputs can hold; this option accepts any
 *      finite input at the cost of that extra rounding.
 * Returns K6ATTN_ERR_INVALID_ARG for an unknown option or a negative value. */
typedef enum {
    K6ATTN_OPT_WAIT_LIMIT_NS = 0,
    K6ATTN_OPT_STRICT_MMA_ORDER = 1,
    K6ATTN_OPT_ROTATE_BF16 = 2
} k6attn_option;
k6attn_status k6attn_set_option(k6attn_t h, k6attn_option opt, long long value);

/* Static description of a status code, and the last error message of the
 * calling thread ("" if none). */
const char *k6attn_status_string(k6attn_status s);
const char *k6attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* K6ATTN_H */
