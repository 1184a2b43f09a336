// k6_bounds.cu -- row bounds for the constant-max softmax.
//
// "Context Parallelism in vLLM Omni Neuron", "Related information": the ring
// kernel `ring_attention_const_max_fwd` takes the softmax max as a runtime
// bound instead of a running max, so no partial output ever needs rescaling
// and the K/V rotation can overlap compute.  The pages name the bound but
// not its formula; this library uses the Cauchy-Schwarz bound
//   M_i = |q_i| * max_j |k_j| / sqrt(d)  >=  max_j q_i . k_j / sqrt(d),
// with the maximum over every key of the (batch, head) pair, so one bound
// serves every K/V chunk.
//
// Two HBM-bound passes: the key-norm maximum per (b, h) (atomic max on the
// float bits, valid because norms are non-negative), then one bound per query
// row.  Half a warp (16 lanes x 8 elements) covers one d = 128 head row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "k6_internal.h"

namespace k6 {

template <typename T>
__device__ __forceinline__ float sumsq8(const void *p) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const T *e = reinterpret_cast<const T *>(&u);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const float x = static_cast<float>(e[k]);
        s = fmaf(x, x, s);
    }
    return s;
}
template <>
__device__ __forceinline__ float sumsq8<float>(const void *p) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
}

// |row| of `rows` head rows of d elements (d / 8 lanes per row, whole rows per warp).
template <typename T>
__device__ __forceinline__ float row_norm(const char *base, long row, int d, int sub, int lanes_per_row) {
    float s = 0.f;
    for (int v = sub; v < d / 8; v += lanes_per_row) s += sumsq8<T>(base + (row * d + v * 8) * sizeof(T));
    for (int o = lanes_per_row / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o, lanes_per_row);
    return sqrtf(s);
}

// kmax[b*H + h] = max over the keys of (b, h) of |k|; keys of two tensors
// (video rows, then joint rows), both [B][rows][H][d].
template <typename T>
__global__ void __launch_bounds__(256) key_norm_max_kernel(const void *k, long Nv, const void *jk, long Nj, int B,
                                                          int H, int d, unsigned *kmax) {
    const int lpr = d / 8 < 32 ? d / 8 : 32;  // lanes per row
    const int rows_per_warp = 32 / lpr;
    const int lane = threadIdx.x & 31, sub = lane % lpr;
    const long warp = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const long total = (long)B * (Nv + Nj) * H;  // head rows
    for (long r0 = warp * rows_per_warp; r0 < total; r0 += nwarps * rows_per_warp) {
        const long r = r0 + lane / lpr;
        const bool live = r < total;
        const long rr = live ? r : total - 1;
        const int h = (int)(rr % H);
        const long bn = rr / H;
        const long n = bn % (Nv + Nj);
        const int b = (int)(bn / (Nv + Nj));
        const char *base;
        long row;
        if (n < Nv) {
            base = static_cast<const char *>(k);
            row = ((long)b * Nv + n) * H + h;
        } else {
            base = static_cast<const char *>(jk);
            row = ((long)b * Nj + (n - Nv)) * H + h;
        }
        const float nrm = row_norm<T>(base, row, d, sub, lpr);
        if (live && sub == 0) atomicMax(kmax + (long)b * H + h, __float_as_uint(nrm));
    }
}

// bound[(b*H + h)*Sq + s] = |q[b][s][h]| * kmax[b*H + h] / sqrt(d)
template <typename T>
__global__ void __launch_bounds__(256) row_bound_kernel(const void *q, long Sq, int B, int H, int d,
                                                       const unsigned *kmax, float inv_sqrt_d, float *bound) {
    const int lpr = d / 8 < 32 ? d / 8 : 32;
    const int rows_per_warp = 32 / lpr;
    const int lane = threadIdx.x & 31, sub = lane % lpr;
    const long warp = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const long total = (long)B * Sq * H;
    for (long r0 = warp * rows_per_warp; r0 < total; r0 += nwarps * rows_per_warp) {
        const long r = r0 + lane / lpr;
        const bool live = r < total;
        const long rr = live ? r : total - 1;  // rr = (b*Sq + s)*H + h
        const int h = (int)(rr % H);
        const long bs = rr / H;
        const long s = bs % Sq;
        const int b = (int)(bs / Sq);
        const float nrm = row_norm<T>(static_cast<const char *>(q), rr, d, sub, lpr);
        if (live && sub == 0)
            bound[((long)b * H + h) * Sq + s] = nrm * __uint_as_float(kmax[(long)b * H + h]) * inv_sqrt_d;
    }
}

cudaError_t launch_row_bounds(const Geom &g, k6attn_dtype qk_dtype, const void *q, const void *k, const void *jk,
                              float *bound, cudaStream_t st) {
    unsigned *kmax = reinterpret_cast<unsigned *>(bound + (size_t)g.B * g.H * g.Sq);
    cudaError_t e = cudaMemsetAsync(kmax, 0, sizeof(unsigned) * g.B * g.H, st);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned blocks = (unsigned)sms * 8;
    const float inv_sqrt_d = 1.0f / sqrtf((float)g.d);
    if (qk_dtype == K6ATTN_F16) {
        key_norm_max_kernel<__half><<<blocks, 256, 0, st>>>(k, g.Nv, jk, g.Nj, g.B, g.H, g.d, kmax);
        row_bound_kernel<__half><<<blocks, 256, 0, st>>>(q, g.Sq, g.B, g.H, g.d, kmax, inv_sqrt_d, bound);
    } else if (qk_dtype == K6ATTN_BF16) {
        key_norm_max_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(k, g.Nv, jk, g.Nj, g.B, g.H, g.d, kmax);
        row_bound_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(q, g.Sq, g.B, g.H, g.d, kmax, inv_sqrt_d, bound);
    } else {
        key_norm_max_kernel<float><<<blocks, 256, 0, st>>>(k, g.Nv, jk, g.Nj, g.B, g.H, g.d, kmax);
        row_bound_kernel<float><<<blocks, 256, 0, st>>>(q, g.Sq, g.B, g.H, g.d, kmax, inv_sqrt_d, bound);
    }
    return cudaGetLastError();
}

}  // namespace k6
