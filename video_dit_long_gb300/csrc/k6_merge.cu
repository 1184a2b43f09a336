// k6_merge.cu -- log-sum-exp merge of per-chunk attention partials.
//
// Ring attention passes K/V chunks between ranks and combines what each
// chunk contributes ("Context Parallelism in vLLM Omni Neuron", sections
// "Ring attention (current implementation)" and "Scaling Properties").  The
// combine (a reading; the pages name it but print no formula):
//   LSE = M + log sum_c exp(LSE_c - M),  M = max_c LSE_c,
//   out = sum_c exp(LSE_c - LSE) * O_c.
//
// HBM-bound: every partial element is read once (streaming loads), every
// output element written once.  One (b, s, h) row of d fp32 per d/4 threads
// (a full warp for d = 128): 16-byte loads, coalesced 512-byte row segments.
#include <cuda_bf16.h>

#include "k6_internal.h"

namespace k6 {

// SHFL (d = 128, n <= 32, one warp per row): lane c holds chunk c's LSE; max and
// sum by warp shuffles, and lane c's weight is broadcast to the accumulation.
template <typename OutT, int D, bool SHFL>
__global__ void __launch_bounds__(256) lse_merge_kernel(int n, long rows, long Sq, int H,
                                                        const float *__restrict__ part_o,
                                                        const float *__restrict__ part_lse, OutT *__restrict__ out,
                                                        float *__restrict__ lse) {
    constexpr int TPR = D / 4;                 // threads per row
    const long o_stride = rows * D;            // floats per chunk
    const long l_stride = rows;                // B*H*Sq
    const int sub = threadIdx.x % TPR;
    long r = (blockIdx.x * (long)blockDim.x + threadIdx.x) / TPR;
    const long step = (long)gridDim.x * blockDim.x / TPR;
    for (; r < rows; r += step) {
        // r enumerates (b, s, h) in output order [B][Sq][H]
        const int h = (int)(r % H);
        const long bs = r / H;
        const long s = bs % Sq;
        const long b = bs / Sq;
        const long li = (b * H + h) * Sq + s;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *po = part_o + r * D + sub * 4;
        float L;
        if constexpr (SHFL) {
            static_assert(TPR == 32, "one warp per row");
            const float lc = sub < n ? __ldg(part_lse + sub * l_stride + li) : -INFINITY;
            float m = lc;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float e = sub < n ? expf(lc - m) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
            L = m + logf(e);
            const float wl = sub < n ? expf(lc - L) : 0.f;
            for (int c0 = 0; c0 < n; c0 += 4) {
                float4 x[4];
#pragma unroll
                for (int u = 0; u < 4; u++)
                    if (c0 + u < n) x[u] = __ldcs(reinterpret_cast<const float4 *>(po + (c0 + u) * o_stride));
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const float wt = __shfl_sync(0xffffffffu, wl, (c0 + u) & 31);
                    if (c0 + u < n) {
                        acc.x += wt * x[u].x;
                        acc.y += wt * x[u].y;
                        acc.z += wt * x[u].z;
                        acc.w += wt * x[u].w;
                    }
                }
            }
        } else {
            float m = -INFINITY;
            for (int c = 0; c < n; c++) m = fmaxf(m, __ldg(part_lse + c * l_stride + li));
            float sum = 0.f;
            for (int c = 0; c < n; c++) sum += expf(__ldg(part_lse + c * l_stride + li) - m);
            L = m + logf(sum);
            // four chunks per pass, loads issued before the arithmetic (eight measured slower)
            for (int c0 = 0; c0 < n; c0 += 4) {
                float4 x[4];
                float wgt[4];
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const int c = c0 + u;
                    if (c < n) {
                        x[u] = __ldcs(reinterpret_cast<const float4 *>(po + c * o_stride));
                        wgt[u] = __ldg(part_lse + c * l_stride + li);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if (c0 + u < n) {
                        const float wt = expf(wgt[u] - L);
                        acc.x += wt * x[u].x;
                        acc.y += wt * x[u].y;
                        acc.z += wt * x[u].z;
                        acc.w += wt * x[u].w;
                    }
                }
            }
        }
        if constexpr (sizeof(OutT) == 2) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            __stcs(reinterpret_cast<uint2 *>(out + r * D + sub * 4), u);
        } else {
            __stcs(reinterpret_cast<float4 *>(out + r * D + sub * 4), acc);
        }
        if (lse && sub == 0) lse[li] = L;
    }
}

cudaError_t launch_lse_merge(const Geom &g, int n, const float *part_o, const float *part_lse, void *out, float *lse,
                             cudaStream_t st) {
    const long rows = (long)g.B * g.Sq * g.H;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    const long tpr = g.d / 4;
    long want = (rows * tpr + threads - 1) / threads;
    long cap = (long)sms * 8;  // 2048 threads per SM resident
    unsigned blocks = (unsigned)(want < cap ? want : cap);
    if (g.d == 128 && n <= 32) {
        if (g.elem == 2)
            lse_merge_kernel<__nv_bfloat16, 128, true><<<blocks, threads, 0, st>>>(
                n, rows, g.Sq, g.H, part_o, part_lse, static_cast<__nv_bfloat16 *>(out), lse);
        else
            lse_merge_kernel<float, 128, true>
                <<<blocks, threads, 0, st>>>(n, rows, g.Sq, g.H, part_o, part_lse, static_cast<float *>(out), lse);
    } else if (g.d == 128) {
        if (g.elem == 2)
            lse_merge_kernel<__nv_bfloat16, 128, false><<<blocks, threads, 0, st>>>(
                n, rows, g.Sq, g.H, part_o, part_lse, static_cast<__nv_bfloat16 *>(out), lse);
        else
            lse_merge_kernel<float, 128, false>
                <<<blocks, threads, 0, st>>>(n, rows, g.Sq, g.H, part_o, part_lse, static_cast<float *>(out), lse);
    } else {
        if (g.elem == 2)
            lse_merge_kernel<__nv_bfloat16, 64, false><<<blocks, threads, 0, st>>>(
                n, rows, g.Sq, g.H, part_o, part_lse, static_cast<__nv_bfloat16 *>(out), lse);
        else
            lse_merge_kernel<float, 64, false>
                <<<blocks, threads, 0, st>>>(n, rows, g.Sq, g.H, part_o, part_lse, static_cast<float *>(out), lse);
    }
    return cudaGetLastError();
}

}  // namespace k6
