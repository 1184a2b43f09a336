// k6_internal.h -- host-side declarations shared by the translation units of
// libk6attn (launchers, geometry, rotary table layout).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "k6attn.h"

namespace k6 {

// Device error word codes (written with atomicCAS, first error wins).
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_RANGE = 2, DEV_LAYOUT = 3 };

// Geometry of one joint attention problem, as the kernels see it.
struct Geom {
    int B, H, d;
    long Nv, Nj, S;          // keys: S = Nv + Nj (video keys, then joint keys)
    long Sq;                 // query rows: S for self-attention, any length for cross-attention
    int grid_t, grid_h, grid_w;
    int axis_dim[3];
    int joint_rope;
    int elem;                // bytes per element (2 bf16, 4 f32)
    k6attn_dtype dtype;      // storage type of q, k, v, out (BF16 or F32)
};

// Offsets (in float2 entries) of the rotary tables inside one buffer.
struct RopeLayout {
    long off[4];             // axis t, h, w, joint
    long total;              // entries
};

RopeLayout rope_layout(const Geom &g);

// Error reporting of the host side (thread-local message).
k6attn_status set_error(k6attn_status s, const char *fmt, ...);
k6attn_status cuda_check(cudaError_t e, const char *what);

// A handle is usable only while its own device is current (its tables and
// error word live there): INVALID_ARG otherwise, and for a null handle.
k6attn_status check_handle(const char *fn, k6attn_t h);

// ---- host helpers shared by the launchers (k6_host.cu) ----

// Unique id of the calling thread's current CUDA context; 0 when none is current.
unsigned long long current_context_id();
// Tensor map over a BSHD tensor [B][rows][H][128] of 2-byte elements (box = 64
// dims x 1 head x 128 rows x 1 batch) or 1-byte elements (box = 128 dims x 1 x
// 128 x 1): 128-byte box rows, 128-byte swizzle, zero fill out of bounds.
bool make_bshd_map(CUtensorMap *m, const void *base, long rows, int H, int B, bool f16, const char **why,
                   int elem_bytes = 2);
// Opt `func` in to `bytes` of dynamic shared memory in the current context
// (once per kernel and context).
cudaError_t set_max_dynamic_smem(const void *func, int bytes);

// ---- launchers (return cudaSuccess or the launch error) ----

cudaError_t launch_rope_tables(const Geom &g, double theta, float2 *tables, cudaStream_t st);

// Optional QK-norm ahead of the rotation: fp32 weights [H*d] for video q rows,
// joint q rows, video k rows and joint k rows (the joint ones default to the
// video ones when null).
struct QkNorm {
    const float *q_w, *jq_w, *k_w, *jk_w;
    float eps;
};

// Rotary embedding of q [B][S][H][d], k [B][Nv][H][d], jk [B][Nj][H][d]
// from src_* (type g.dtype) into dst_* (type out_dtype; dst may equal src
// when the types match).  Writing F16, a value that is not finite in fp16
// sets *err to DEV_RANGE.
cudaError_t launch_rope_qk(const Geom &g, const float2 *tables, const void *src_q, void *dst_q, const void *src_k,
                           void *dst_k, const void *src_jk, void *dst_jk, k6attn_dtype out_dtype, int *err,
                           cudaStream_t st, const QkNorm *norm = nullptr);

// Merge of n partials of problem g (P = 1), or of the P*B problems of g.H/P
// heads of a P-way head split of g, written to g's sequence layout.
// Rotary of q/k/joint_k (into qk_out: BF16, F16 or E4M3) and the P-way
// sequence->head split of q, k, joint_k, v, joint_v (index order) of a bf16
// d = 128 problem g: dst[t] is [P][B][rows_t][H/P][128].
cudaError_t launch_rope_split(const Geom &g, const float2 *tables, const void *const src[5], void *const dst[5],
                              int P, k6attn_dtype qk_out, int *err, cudaStream_t st);

cudaError_t launch_lse_merge(const Geom &g, int n, const float *part_o, const float *part_lse, void *out, float *lse,
                             cudaStream_t st, int P = 1);

cudaError_t launch_relayout(const void *src, void *dst, int B, long S, int H, int d, int elem_bytes, int P,
                            int direction, cudaStream_t st);

// fp32 attention (SIMT): per chunk c writes out_c [B][S][H][d] and lse_c
// [B][H][S], at out + c*o_stride / lse + c*l_stride.
cudaError_t launch_attn_f32(const Geom &g, const float *q, const float *k, const float *v, const float *jk,
                            const float *jv, int n_chunks, float *out, size_t o_stride, float *lse, size_t l_stride,
                            cudaStream_t st);

// bf16 attention on tcgen05 tensor cores.  n_chunks == 1: out is bf16
// [B][S][H][d]; n_chunks > 1: out is fp32 partials [n][B][S][H][d].
// lse is fp32 [n][B][H][S] (may be null when n_chunks == 1).
struct AttnTcOptions {
    unsigned long long wait_limit_ns;
    int *err;
    int strict_order;        // accepted; the kernel already waits for P.V before reusing its TMEM
    int qk_f16;              // 1: q/k/joint_k are fp16 (Q.K^T in fp16), else bf16
    const float *row_bound = nullptr;  // constant-max softmax bounds [B][H][Sq] (natural-log units), or null
    int qk8 = 0;             // 1: q/k/joint_k are e4m3 (Q.K^T on kind::f8f6f4)
    int group = 0;           // chunks per CTA (divides n_chunks); 0: the library's choice, chunk_group()
    int merge = 0;           // 1: each CTA's group of chunks leaves one partial (n_chunks / group partials)
};

// Chunks per CTA the library picks for n_chunks K/V chunks of problem g on the
// current device: the largest divisor of n_chunks up to 4 that still leaves at
// least four waves of CTAs (short query ranges keep one chunk per CTA).
int chunk_group(const Geom &g, int n_chunks);

// Constant-max bounds: bound[(b*H + h)*Sq + s] = |q| * max|k| / sqrt(d);
// bound must hold B*H*Sq + B*H floats (the tail is the key-norm maximum).
cudaError_t launch_row_bounds(const Geom &g, k6attn_dtype qk_dtype, const void *q, const void *k, const void *jk,
                              float *bound, cudaStream_t st);
// One CTA per 128-row Q tile and group of chunks (k6_attn_single.cu).
cudaError_t launch_attn_tc_single(const Geom &g, const void *q, const void *k, const void *v, const void *jk,
                                  const void *jv, int n_chunks, void *out, float *lse, const AttnTcOptions &opt,
                                  cudaStream_t st, const char **why);

// Backward pass (bf16 v/out/dout, q/k bf16 or fp16, d = 128): the pre-pass
// into LD [B][H][S] = {lse * log2(e), D_i}, then the dq kernel and the dk/dv kernel.
cudaError_t launch_attn_bwd(const Geom &g, bool qk_f16, const void *q, const void *k, const void *v, const void *jk,
                            const void *jv, const void *out, const void *dout, const float *lse, float2 *LD, float *dq,
                            float *dk, float *dv, float *djk, float *djv, unsigned long long wait_limit_ns, int *err,
                            cudaStream_t st, const char **why);

}  // namespace k6
