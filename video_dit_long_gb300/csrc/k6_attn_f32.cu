// k6_attn_f32.cu -- fp32 joint-sequence attention on the CUDA cores (SIMT).
//
// Full non-causal attention softmax(q k^T / sqrt(d)) v over the joint
// sequence (xDiT PR #586, "How?" and the USP `_attention` call; "Context
// Parallelism in vLLM Omni Neuron", "Self-Attention with Context
// Parallelism"), per K/V chunk with an online softmax, writing the chunk's
// output and log-sum-exp ("Ring attention (current implementation)").
//
// fp32 end to end (fp32 products, fp32 softmax with expf): the fp32 workload
// asks for 1e-4 agreement, which tf32 tensor-core products cannot give.
// Each CTA owns 128 query rows of one (batch, head, chunk); 64 head dims per
// thread (one thread per row for d = 64, two for d = 128, combined with a
// shuffle); K/V tiles of 32 keys staged in shared memory.
#include "k6_internal.h"

namespace k6 {

constexpr int F32_ROWS = 128;
constexpr int F32_KEYS = 32;

template <int D>
__global__ void __launch_bounds__(F32_ROWS *(D / 64)) attn_f32_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    const float *__restrict__ jk, const float *__restrict__ jv, long Sq, long S, long Nv, int H, int n_chunks,
    float *__restrict__ out, size_t o_stride, float *__restrict__ lse, size_t l_stride, float scale) {
    constexpr int TPR = D / 64;  // threads per query row
    __shared__ float ks[F32_KEYS][D];
    __shared__ float vs[F32_KEYS][D];
    const int h = blockIdx.y;
    const int b = blockIdx.z / n_chunks;
    const int c = blockIdx.z % n_chunks;
    const long row = (long)blockIdx.x * F32_ROWS + threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;  // which 64 dims this thread owns
    const long L = S / n_chunks;
    const long kb = (long)c * L, ke = kb + L;
    const long Nj = S - Nv;

    float qr[64], o[64];
    const bool live = row < Sq;
    const float *qp = q + (((long)b * Sq + (live ? row : 0)) * H + h) * D + part * 64;
#pragma unroll
    for (int e = 0; e < 64; e++) {
        qr[e] = live ? qp[e] : 0.f;
        o[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    for (long t0 = kb; t0 < ke; t0 += F32_KEYS) {
        __syncthreads();
        for (int i = threadIdx.x; i < F32_KEYS * D / 4; i += blockDim.x) {
            const int key = i / (D / 4), e4 = i % (D / 4);
            const long n = t0 + key;
            float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
            if (n < ke) {
                const float *kp, *vp;
                if (n < Nv) {
                    kp = k + (((long)b * Nv + n) * H + h) * D;
                    vp = v + (((long)b * Nv + n) * H + h) * D;
                } else {
                    kp = jk + (((long)b * Nj + (n - Nv)) * H + h) * D;
                    vp = jv + (((long)b * Nj + (n - Nv)) * H + h) * D;
                }
                kx = reinterpret_cast<const float4 *>(kp)[e4];
                vx = reinterpret_cast<const float4 *>(vp)[e4];
            }
            reinterpret_cast<float4 *>(&ks[key][0])[e4] = kx;
            reinterpret_cast<float4 *>(&vs[key][0])[e4] = vx;
        }
        __syncthreads();
        const int nk = (int)((ke - t0) < F32_KEYS ? (ke - t0) : F32_KEYS);
        float s[F32_KEYS];
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < F32_KEYS; j++) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 64; e++) acc = fmaf(qr[e], ks[j][part * 64 + e], acc);
            if (TPR == 2) acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            s[j] = j < nk ? acc * scale : -INFINITY;
            mt = fmaxf(mt, s[j]);
        }
        const float mn = fmaxf(m, mt);
        const float alpha = expf(m - mn);  // m = -inf on the first tile: alpha = 0
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 64; e++) o[e] *= alpha;
#pragma unroll
        for (int j = 0; j < F32_KEYS; j++) {
            const float p = expf(s[j] - mn);
            l += p;
#pragma unroll
            for (int e = 0; e < 64; e++) o[e] = fmaf(p, vs[j][part * 64 + e], o[e]);
        }
        m = mn;
    }
    if (!live) return;
    const float inv = 1.f / l;
    float *op = out + c * o_stride + (((long)b * Sq + row) * H + h) * D + part * 64;
#pragma unroll
    for (int e = 0; e < 64; e += 4)
        *reinterpret_cast<float4 *>(op + e) = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
    if (lse && part == 0) lse[c * l_stride + ((long)b * H + h) * Sq + row] = m + logf(l);
}

cudaError_t launch_attn_f32(const Geom &g, const float *q, const float *k, const float *v, const float *jk,
                            const float *jv, int n_chunks, float *out, size_t o_stride, float *lse, size_t l_stride,
                            cudaStream_t st) {
    dim3 grid((unsigned)((g.Sq + F32_ROWS - 1) / F32_ROWS), (unsigned)g.H, (unsigned)(g.B * n_chunks));
    const float scale = 1.0f / sqrtf((float)g.d);
    if (g.d == 64)
        attn_f32_kernel<64><<<grid, F32_ROWS, 0, st>>>(q, k, v, jk, jv, g.Sq, g.S, g.Nv, g.H, n_chunks, out, o_stride, lse,
                                                       l_stride, scale);
    else
        attn_f32_kernel<128><<<grid, F32_ROWS * 2, 0, st>>>(q, k, v, jk, jv, g.Sq, g.S, g.Nv, g.H, n_chunks, out, o_stride,
                                                            lse, l_stride, scale);
    return cudaGetLastError();
}

}  // namespace k6
