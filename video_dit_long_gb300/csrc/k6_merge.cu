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
//
// The partials may come from the head-partitioned layout of a P-way Ulysses
// split (P*B problems of H/P heads, xDiT PR #586 USP dispatch listing,
// `_ft_c_output_all_to_all`): the merge then writes each row straight to its
// place in the sequence layout [B][Sq][H][d] (head p*H/P + hh of batch b for
// problem p*B + b), so the head->seq relayout of the output costs no pass of
// its own.  P = 1 is the plain merge.
#include <cuda_bf16.h>

#include "k6_internal.h"

namespace k6 {

// SHFL (d = 128, n <= 32, one warp per row): lane c holds chunk c's LSE; max and
// sum by warp shuffles, and lane c's weight is broadcast to the accumulation.
// rows = P*B*Sq*Hl partial rows; the partials are [n][P*B][Sq][Hl][D] and
// [n][P*B][Hl][Sq], the outputs [B][Sq][P*Hl][D] and [B][P*Hl][Sq].
template <typename OutT, int D, bool SHFL>
__global__ void __launch_bounds__(256) lse_merge_kernel(int n, long rows, long Sq, int Hl, int B, int P,
                                                        const float *__restrict__ part_o,
                                                        const float *__restrict__ part_lse, OutT *__restrict__ out,
                                                        float *__restrict__ lse) {
    constexpr int TPR = D / 4;                 // threads per row
    const long o_stride = rows * D;            // floats per chunk
    const long l_stride = rows;                // P*B*Hl*Sq
    const int sub = threadIdx.x % TPR;
    long r = (blockIdx.x * (long)blockDim.x + threadIdx.x) / TPR;
    const long step = (long)gridDim.x * blockDim.x / TPR;
    const int H = Hl * P;
    for (; r < rows; r += step) {
        // r enumerates (problem, s, hh) in partial order [P*B][Sq][Hl]; 32-bit
        // index arithmetic (the host keeps B*Sq*H below 2^31)
        const unsigned ru = (unsigned)r;
        const unsigned hh = ru % (unsigned)Hl;
        const unsigned t = ru / (unsigned)Hl;
        const unsigned s = t % (unsigned)Sq;
        const unsigned pb = t / (unsigned)Sq;
        const long li = ((long)pb * Hl + hh) * Sq + s;      // partial LSE index
        const unsigned b = pb % (unsigned)B;
        const unsigned h = (pb / (unsigned)B) * Hl + hh;     // head in the full layout
        const long orow = ((long)b * Sq + s) * H + h;        // output row [B][Sq][H]
        const long lo = ((long)b * H + h) * Sq + s;          // output LSE index [B][H][Sq]
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
            __stcs(reinterpret_cast<uint2 *>(out + orow * D + sub * 4), u);
        } else {
            __stcs(reinterpret_cast<float4 *>(out + orow * D + sub * 4), acc);
        }
        if (lse && sub == 0) lse[lo] = L;
    }
}

// Few partials (N <= 4, d = 128): with one warp per row a lane would have only
// N 16-byte loads in flight, too few to cover HBM latency.  Here a warp takes R
// consecutive rows at a time (N * R = 8 loads of 16 bytes per lane for N >= 2,
// 4 for N = 1, all issued before any arithmetic), in partial order
// [P*B][Sq][Hl], so the partial
// outputs stream through HBM in address order; the partial LSEs ([P*B][Hl][Sq],
// a few MB) are read with a stride and served mostly from L2.  Each lane forms
// the row's LSE from the N partial LSEs itself (warp-wide broadcast reads).
// Index arithmetic is 32-bit: 64-bit divisions per row made the kernel
// instruction-bound (measured: 60 % SM throughput at 52 % of DRAM bandwidth).
template <typename OutT, int N, int R>
__global__ void __launch_bounds__(256, 3) lse_merge_few_kernel(long rows, long Sq, int Hl, int B, int P,
                                                            const float *__restrict__ part_o,
                                                            const float *__restrict__ part_lse,
                                                            OutT *__restrict__ out, float *__restrict__ lse) {
    constexpr int D = 128;
    const int sub = threadIdx.x & 31;
    const long warp = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const long o_stride = rows * D, l_stride = rows;
    const int H = Hl * P;
    for (long r0 = warp * R; r0 < rows; r0 += nwarps * R) {
        float4 x[R][N];
        float lc[R][N];
        long orow[R], lo[R];
#pragma unroll
        for (int rr = 0; rr < R; rr++) {
            // a clamped row is computed, not stored; 32-bit index arithmetic (B*Sq*H < 2^31)
            const unsigned r = (unsigned)(r0 + rr < rows ? r0 + rr : rows - 1);
            const unsigned hh = r % (unsigned)Hl;
            const unsigned t = r / (unsigned)Hl;
            const unsigned s = t % (unsigned)Sq;
            const unsigned pb = t / (unsigned)Sq;
            const long li = ((long)pb * Hl + hh) * Sq + s;       // partial LSE [P*B][Hl][Sq]
            const unsigned b = pb % (unsigned)B;
            const unsigned h = (pb / (unsigned)B) * Hl + hh;
            orow[rr] = ((long)b * Sq + s) * H + h;               // output row [B][Sq][H]
            lo[rr] = ((long)b * H + h) * Sq + s;                 // output LSE [B][H][Sq]
#pragma unroll
            for (int c = 0; c < N; c++)
                x[rr][c] = __ldcs(reinterpret_cast<const float4 *>(part_o + c * o_stride + (long)r * D) + sub);
#pragma unroll
            for (int c = 0; c < N; c++) lc[rr][c] = __ldg(part_lse + c * l_stride + li);
        }
#pragma unroll
        for (int rr = 0; rr < R; rr++) {
            float m = lc[rr][0];
#pragma unroll
            for (int c = 1; c < N; c++) m = fmaxf(m, lc[rr][c]);
            float e = 0.f;
#pragma unroll
            for (int c = 0; c < N; c++) e += expf(lc[rr][c] - m);
            const float L = m + logf(e);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < N; c++) {
                const float wt = expf(lc[rr][c] - L);
                acc.x += wt * x[rr][c].x;
                acc.y += wt * x[rr][c].y;
                acc.z += wt * x[rr][c].z;
                acc.w += wt * x[rr][c].w;
            }
            if (r0 + rr >= rows) continue;
            if constexpr (sizeof(OutT) == 2) {
                __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
                __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t *>(&lo2);
                u.y = *reinterpret_cast<uint32_t *>(&hi2);
                __stcs(reinterpret_cast<uint2 *>(out + orow[rr] * D) + sub, u);
            } else {
                __stcs(reinterpret_cast<float4 *>(out + orow[rr] * D) + sub, acc);
            }
            if (lse && sub == 0) lse[lo[rr]] = L;
        }
    }
}

cudaError_t launch_lse_merge(const Geom &g, int n, const float *part_o, const float *part_lse, void *out, float *lse,
                             cudaStream_t st, int P) {
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
    const int Hl = g.H / P;
    auto launch = [&](auto kernel, auto *o) {
        kernel<<<blocks, threads, 0, st>>>(n, rows, g.Sq, Hl, g.B, P, part_o, part_lse, o, lse);
    };
    __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(out);
    float *of = static_cast<float *>(out);
    if (g.d == 128 && n <= 4) {
        // R rows per warp pass; the grid covers the rows once where it can
        auto few = [&](auto kernel, auto *o, int R) {
            long w = (rows + R - 1) / R;  // warps wanted
            long b = (w + 7) / 8;
            unsigned nb = (unsigned)(b < cap ? b : cap);
            kernel<<<nb, threads, 0, st>>>(rows, g.Sq, Hl, g.B, P, part_o, part_lse, o, lse);
        };
        if (g.elem == 2) {
            if (n == 1) few(lse_merge_few_kernel<__nv_bfloat16, 1, 4>, ob, 4);
            else if (n == 2) few(lse_merge_few_kernel<__nv_bfloat16, 2, 4>, ob, 4);
            else if (n == 3) few(lse_merge_few_kernel<__nv_bfloat16, 3, 2>, ob, 2);
            else few(lse_merge_few_kernel<__nv_bfloat16, 4, 2>, ob, 2);
        } else {
            if (n == 1) few(lse_merge_few_kernel<float, 1, 4>, of, 4);
            else if (n == 2) few(lse_merge_few_kernel<float, 2, 4>, of, 4);
            else if (n == 3) few(lse_merge_few_kernel<float, 3, 2>, of, 2);
            else few(lse_merge_few_kernel<float, 4, 2>, of, 2);
        }
    } else if (g.d == 128 && n <= 32) {
        if (g.elem == 2) launch(lse_merge_kernel<__nv_bfloat16, 128, true>, ob);
        else launch(lse_merge_kernel<float, 128, true>, of);
    } else if (g.d == 128) {
        if (g.elem == 2) launch(lse_merge_kernel<__nv_bfloat16, 128, false>, ob);
        else launch(lse_merge_kernel<float, 128, false>, of);
    } else {
        if (g.elem == 2) launch(lse_merge_kernel<__nv_bfloat16, 64, false>, ob);
        else launch(lse_merge_kernel<float, 64, false>, of);
    }
    return cudaGetLastError();
}

}  // namespace k6
