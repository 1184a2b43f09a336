// k6_relayout.cu -- sequence-partitioned <-> head-partitioned relayout.
//
// Ulysses sequence parallelism moves Q, K and V from "each rank holds a token
// range, all heads" to "each rank holds all tokens, a head range" with an
// all-to-all, and moves the output back with another (xDiT PR #586, USP
// dispatch listing: `_ft_c_input_all_to_all`, `_ft_c_output_all_to_all`;
// "Context Parallelism in vLLM Omni Neuron", "Comparison with Other CP
// Strategies": two all-to-alls, num_heads % cp_size == 0).  On one GPU the
// exchange is a permutation of HBM:
//   head[p][b][r*Sl + s][hh][e] = seq[r][b][s][p*Hl + hh][e],  Sl = S/P, Hl = H/P.
//
// Every head-buffer row (p, b, token) is one contiguous run of Hl*d elements,
// and so is its source.  One warp copies one run per iteration with 16-byte
// vectors (narrower only when the run is not a multiple of 16 bytes), so the
// index arithmetic (32-bit) is paid once per run, not per element; four runs
// per warp-iteration with every load issued before the stores keep enough
// bytes in flight.  Pure byte moves: bit-exact by construction.
#include <cuda_runtime.h>

#include "k6_internal.h"

namespace k6 {

template <typename V>
__global__ void __launch_bounds__(256) relayout_kernel(const char *__restrict__ src, char *__restrict__ dst,
                                                       unsigned B, unsigned S, unsigned Sl, unsigned H, unsigned Hl,
                                                       unsigned run_bytes, unsigned rows, int direction) {
    constexpr int kRows = 4;     // runs per warp-iteration
    constexpr int kPerLane = 2;  // words per lane per run and pass
    const unsigned lane = threadIdx.x & 31;
    const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
    const unsigned nvec = run_bytes / sizeof(V);
    const unsigned long long row_bytes_seq = (unsigned long long)run_bytes * (H / Hl);  // H*d*eb
    for (unsigned hr0 = warp * kRows; hr0 < rows; hr0 += nwarps * kRows) {
        const V *from[kRows];
        V *to[kRows];
#pragma unroll
        for (int i = 0; i < kRows; i++) {
            // hr = (p*B + b)*S + token
            const unsigned hr = min(hr0 + i, rows - 1);
            const unsigned token = hr % S;
            const unsigned pb = hr / S;
            const unsigned b = pb % B;
            const unsigned p = pb / B;
            const unsigned r = token / Sl;
            const unsigned s = token % Sl;
            const unsigned long long head_off = (unsigned long long)hr * run_bytes;
            const unsigned long long seq_off =
                ((unsigned long long)(r * B + b) * Sl + s) * row_bytes_seq + (unsigned long long)p * run_bytes;
            from[i] = reinterpret_cast<const V *>(src + (direction == 0 ? seq_off : head_off));
            to[i] = reinterpret_cast<V *>(dst + (direction == 0 ? head_off : seq_off));
        }
        const int live = (int)min((unsigned)kRows, rows - hr0);
        for (unsigned base = 0; base < nvec; base += 32 * kPerLane) {
            V x[kRows][kPerLane];
#pragma unroll
            for (int i = 0; i < kRows; i++)
#pragma unroll
                for (int u = 0; u < kPerLane; u++) {
                    const unsigned k = base + u * 32 + lane;
                    if (i < live && k < nvec) x[i][u] = __ldcs(from[i] + k);
                }
#pragma unroll
            for (int i = 0; i < kRows; i++)
#pragma unroll
                for (int u = 0; u < kPerLane; u++) {
                    const unsigned k = base + u * 32 + lane;
                    if (i < live && k < nvec) __stcs(to[i] + k, x[i][u]);
                }
        }
    }
}

// The relayout kernel moves 16-, 4- or 2-byte words.
template <typename V>
static cudaError_t launch_relayout_t(const void *src, void *dst, int B, long S, int H, int d, int elem_bytes, int P,
                                     int direction, cudaStream_t st) {
    const unsigned Sl = (unsigned)(S / P), Hl = (unsigned)(H / P);
    const unsigned run_bytes = Hl * (unsigned)d * (unsigned)elem_bytes;
    const unsigned rows = (unsigned)P * (unsigned)B * (unsigned)S;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned runs_per_block = 8 * 4;  // 8 warps x 4 runs
    unsigned blocks = (rows + runs_per_block - 1) / runs_per_block;
    unsigned cap = (unsigned)sms * 8;
    if (blocks > cap) blocks = cap;
    relayout_kernel<V><<<blocks, 256, 0, st>>>(static_cast<const char *>(src), static_cast<char *>(dst), (unsigned)B,
                                                (unsigned)S, Sl, (unsigned)H, Hl, run_bytes, rows, direction);
    return cudaGetLastError();
}

cudaError_t launch_relayout(const void *src, void *dst, int B, long S, int H, int d, int elem_bytes, int P,
                            int direction, cudaStream_t st) {
    if ((long)P * B * S == 0) return cudaSuccess;
    const unsigned run_bytes = (unsigned)(H / P) * (unsigned)d * (unsigned)elem_bytes;
    const uintptr_t align = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
    if (run_bytes % 16 == 0 && align % 16 == 0)
        return launch_relayout_t<uint4>(src, dst, B, S, H, d, elem_bytes, P, direction, st);
    if (run_bytes % 4 == 0 && align % 4 == 0)
        return launch_relayout_t<uint32_t>(src, dst, B, S, H, d, elem_bytes, P, direction, st);
    return launch_relayout_t<uint16_t>(src, dst, B, S, H, d, elem_bytes, P, direction, st);
}

}  // namespace k6
