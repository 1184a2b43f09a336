// k6_attn_bwd.cu -- backward pass of the joint-sequence attention on tcgen05.
//
// The pages describe inference only; the gradients are the plain chain rule of
// O = softmax(S) V with S = Q K^T / sqrt(d), on the rotated q and k:
//   D_i  = sum_e dO_ie O_ie                 (pre-pass, HBM-bound)
//   P    = exp(S - LSE)                     (LSE from the forward pass)
//   dP   = dO V^T,   dS = P o (dP - D)
//   dV   = P^T dO,   dK = dS^T Q / sqrt(d), dQ = dS K / sqrt(d)
// over the full key range (video keys, then joint keys) of each (batch, head).
//
// Two kernels, each with one stationary 128-row tile per CTA and the other
// operand streamed through a two-slot TMA ring:
//   dq kernel  (Q, dO stationary, K/V streamed): S = Q K_j^T and dP = dO V_j^T
//              (SS) into tensor memory; four warps turn each row into dS and
//              store it (Q/K operand type) over the first 64 columns of S;
//              dQ += dS K_j (TS, K_j MN-major).  Columns: S | dP | dQ.
//   dkv kernel (K, V stationary, Q/dO streamed): S^T = K Q_i^T, dP^T = V dO_i^T
//              (SS); each thread (one key) turns its row into P^T and dS^T
//              (stored over S^T and dP^T); dV += P^T dO_i, dK += dS^T Q_i
//              (TS).  Columns: S^T | dP^T | dV | dK (all 512).
// One elected thread issues the MMAs; one warp drives TMA; all waits are
// bounded like the forward kernel's.  Gradients are written in fp32.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "k6_device.cuh"
#include "k6_internal.h"

namespace k6 {

namespace bw {
constexpr int D = 128, BM = 128;
constexpr int PANEL = BM * 64 * 2;
constexpr int TILE = 2 * PANEL;             // 32 KB: 128 rows x 128 dims, 16-bit
constexpr int SMEM_STAT = 0;                // two stationary tiles
constexpr int SMEM_RING = 2 * TILE;         // two slots of two tiles each
constexpr int SMEM_BAR = SMEM_RING + 2 * 2 * TILE;
constexpr int NBAR = 1 + 2 + 2 + 1 + 1 + 1 + 1;  // stat_full, ld_full[2], ld_empty[2], s_full, ds_full, acc_done, drain
constexpr int SMEM_ALLOC = SMEM_BAR + NBAR * 8 + 64 + 1024;  // barriers, TMEM slot, abort flag, alignment
constexpr int THREADS = 192;                // warps 0-3 compute, 4 TMA, 5 MMA
constexpr unsigned long long DRAIN_NS = 1000000000ull;
}  // namespace bw

struct BwParams {
    long S, Nv, Nj;
    int H, q_tiles, kv_tiles_v, kv_tiles_j;
    float scale_log2, scale;                // log2(e)/sqrt(d), 1/sqrt(d)
    const float *lse;                       // [B][H][S] natural log
    const float *Dsum;                      // [B][H][S]
    float *dq, *dk, *dv, *djk, *djv;        // fp32 gradients
    uint32_t idesc_qk, idesc_bf16, idesc_ds_q, idesc_ds_k;
    int ds_f16;                             // dS stored as fp16 (q/k are fp16) or bf16
    unsigned long long wait_limit_ns;
    int *err;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool f16) {
    if (f16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    return pack_bf16x2(lo, hi);
}

// ------------------------------------------------------------- pre-pass D

__global__ void __launch_bounds__(256) bwd_dsum_kernel(const __nv_bfloat16 *__restrict__ out,
                                                      const __nv_bfloat16 *__restrict__ dout, long S, int H, int B,
                                                      float *__restrict__ Dsum) {
    const int lane = threadIdx.x & 31, sub = lane & 15;
    const long warp = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const long rows = (long)B * S * H;
    for (long r0 = warp * 2; r0 < rows; r0 += nwarps * 2) {
        const long r = r0 + (lane >> 4);
        const long rr = r < rows ? r : rows - 1;
        const uint4 a = reinterpret_cast<const uint4 *>(out + rr * bw::D)[sub];
        const uint4 b = reinterpret_cast<const uint4 *>(dout + rr * bw::D)[sub];
        const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
        const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float2 fx = __bfloat1622float2(x[k]), fy = __bfloat1622float2(y[k]);
            s = fmaf(fx.x, fy.x, s);
            s = fmaf(fx.y, fy.y, s);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o, 16);
        if (r < rows && sub == 0) {
            const int h = (int)(r % H);
            const long bs = r / H;
            Dsum[((bs / S) * H + h) * S + bs % S] = s;
        }
    }
}

// Shared set-up of both kernels: barriers, tensor memory, abort flag.
struct BwShared {
    uint64_t *stat_full, *ld_full, *ld_empty, *s_full, *ds_full, *acc_done, *drain;
    uint32_t *tmem_slot;
    volatile int *abort;
};

__device__ __forceinline__ BwShared bw_setup(uint8_t *smem) {
    BwShared b;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + bw::SMEM_BAR);
    b.stat_full = bars;
    b.ld_full = bars + 1;
    b.ld_empty = bars + 3;
    b.s_full = bars + 5;
    b.ds_full = bars + 6;
    b.acc_done = bars + 7;
    b.drain = bars + 8;
    b.tmem_slot = reinterpret_cast<uint32_t *>(bars + bw::NBAR);
    b.abort = reinterpret_cast<volatile int *>(b.tmem_slot + 1);
    if (threadIdx.x == 0) {
        mbar_init(b.stat_full, 1);
        for (int s = 0; s < 2; s++) {
            mbar_init(&b.ld_full[s], 1);
            mbar_init(&b.ld_empty[s], 1);
        }
        mbar_init(b.s_full, 1);
        mbar_init(b.ds_full, 128);
        mbar_init(b.acc_done, 1);
        mbar_init(b.drain, 1);
        *b.abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x / 32 == 5) {
        tmem_alloc(b.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return b;
}

__device__ __forceinline__ void bw_teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x / 32 == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Streamed tile t of the key range: which map (0 video, 1 joint) and first row.
__device__ __forceinline__ void kv_tile(const BwParams &p, int t, int &map, int &row) {
    if (t < p.kv_tiles_v) {
        map = 0;
        row = t * bw::BM;
    } else {
        map = 1;
        row = (t - p.kv_tiles_v) * bw::BM;
    }
}

// ------------------------------------------------------------------ dq kernel

__global__ void __launch_bounds__(bw::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_jk, const __grid_constant__ CUtensorMap tm_jv,
                  const BwParams p) {
    using namespace bw;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BwShared sh = bw_setup(smem);
    const uint32_t tmem = *sh.tmem_slot;
    const WaitCtx w{p.wait_limit_ns, p.err, sh.abort};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = blockIdx.x % p.q_tiles;
    const int h = (blockIdx.x / p.q_tiles) % p.H;
    const int b = blockIdx.x / (p.q_tiles * p.H);
    const int q0 = qt * BM;
    const int T = p.kv_tiles_v + p.kv_tiles_j;

    if (warp == 4) {
        if (lane == 0) {
            mbar_arrive_expect_tx(sh.stat_full, 2 * TILE);
            for (int half = 0; half < 2; half++) {
                tma_load_4d(smem + SMEM_STAT + half * PANEL, &tm_q, sh.stat_full, half * 64, h, q0, b);
                tma_load_4d(smem + SMEM_STAT + TILE + half * PANEL, &tm_do, sh.stat_full, half * 64, h, q0, b);
            }
            int issued = 0;
            for (int t = 0; t < T; t++) {
                const int slot = t & 1;
                if (!mbar_wait(&sh.ld_empty[slot], ((t >> 1) & 1) ^ 1, w)) break;
                int map, row;
                kv_tile(p, t, map, row);
                mbar_arrive_expect_tx(&sh.ld_full[slot], 2 * TILE);
                uint8_t *dst = smem + SMEM_RING + slot * 2 * TILE;
                for (int half = 0; half < 2; half++) {
                    tma_load_4d(dst + half * PANEL, map ? &tm_jk : &tm_k, &sh.ld_full[slot], half * 64, h, row, b);
                    tma_load_4d(dst + TILE + half * PANEL, map ? &tm_jv : &tm_v, &sh.ld_full[slot], half * 64, h,
                                row, b);
                }
                issued++;
            }
            mbar_drain(sh.stat_full, 0, DRAIN_NS);
            for (int t = issued > 2 ? issued - 2 : 0; t < issued; t++)
                mbar_drain(&sh.ld_full[t & 1], (t >> 1) & 1, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t tS = tmem, tP = tmem + 128, tA = tmem + 256;
            const uint64_t dq0 = smem_desc_sw128(smem_u32(smem + SMEM_STAT), 16, 1024);        // Q (K-major)
            const uint64_t ddo = dq0 + (uint64_t)(TILE >> 4);                               // dO (K-major)
            const uint64_t dring = smem_desc_sw128(smem_u32(smem + SMEM_RING), 16, 1024);    // K / V (K-major)
            const uint64_t dring_mn = smem_desc_sw128(smem_u32(smem + SMEM_RING), PANEL, 1024);  // K (MN-major)
            bool ok = mbar_wait(sh.stat_full, 0, w);
            for (int t = 0; t < T && ok; t++) {
                const int slot = t & 1;
                if (!(ok = mbar_wait(&sh.ld_full[slot], (t >> 1) & 1, w))) break;
                tc_fence_after();
                const uint64_t kdesc = dring + (uint64_t)((slot * 2 * TILE) >> 4);
                const uint64_t vdesc = kdesc + (uint64_t)(TILE >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    const uint64_t off = (uint64_t)((kk >> 2) * PANEL + (kk & 3) * 32) >> 4;
                    mma_ss(tS, dq0 + off, kdesc + off, p.idesc_qk, kk > 0);     // S = Q K^T
                    mma_ss(tP, ddo + off, vdesc + off, p.idesc_bf16, kk > 0);   // dP = dO V^T
                }
                tc_commit(sh.s_full);
                if (!(ok = mbar_wait(sh.ds_full, t & 1, w))) break;
                tc_fence_after();
                const uint64_t kmn = dring_mn + (uint64_t)((slot * 2 * TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < BM / 16; kk++)
                    mma_ts(tA, tS + kk * 8, kmn + (uint64_t)((kk * 16 * 128) >> 4), p.idesc_ds_k,
                           (t > 0 || kk > 0) ? 1u : 0u);                            // dQ += dS K
                tc_commit(&sh.ld_empty[slot]);
            }
            tc_commit(sh.acc_done);
            tc_commit(sh.drain);
            mbar_drain(sh.drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ compute: one query row per thread
        const int r = threadIdx.x;
        const uint32_t lb = tmem + ((uint32_t)(32 * warp) << 16);
        const long grow = (long)q0 + r;
        const bool live = grow < p.S;
        const long li = ((long)b * p.H + h) * p.S + (live ? grow : 0);
        const float lse2 = live ? p.lse[li] * 1.4426950408889634f : 0.f;
        const float Di = live ? p.Dsum[li] : 0.f;
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int t = 0; t < T; t++) {
            if (!mbar_wait(sh.s_full, t & 1, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t sv[32], pv[32], ds[16];
                tmem_ld32(lb + c * 32, sv);
                tmem_ld32(lb + 128 + c * 32, pv);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const float p0 = ex2(fmaf(__uint_as_float(sv[k]), sl2, -lse2));
                    const float p1 = ex2(fmaf(__uint_as_float(sv[k + 1]), sl2, -lse2));
                    ds[k / 2] = pack2(p0 * (__uint_as_float(pv[k]) - Di), p1 * (__uint_as_float(pv[k + 1]) - Di),
                                      p.ds_f16);
                }
                tmem_st16(lb + c * 16, ds);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(sh.ds_full);
        }
        if (ok && mbar_wait(sh.acc_done, 0, w)) {
            tc_fence_after();
            float *dst = p.dq + (((long)b * p.S + (live ? grow : 0)) * p.H + h) * D;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t o[32];
                tmem_ld32(lb + 256 + c * 32, o);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4 *>(dst + c * 32 + k) =
                            make_float4(__uint_as_float(o[k]) * p.scale, __uint_as_float(o[k + 1]) * p.scale,
                                        __uint_as_float(o[k + 2]) * p.scale, __uint_as_float(o[k + 3]) * p.scale);
                }
            }
        }
    }
    bw_teardown(tmem);
}

// ----------------------------------------------------------------- dkv kernel

__global__ void __launch_bounds__(bw::THREADS, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_jk, const __grid_constant__ CUtensorMap tm_jv,
                   const BwParams p) {
    using namespace bw;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BwShared sh = bw_setup(smem);
    const uint32_t tmem = *sh.tmem_slot;
    const WaitCtx w{p.wait_limit_ns, p.err, sh.abort};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int KT = p.kv_tiles_v + p.kv_tiles_j;
    const int kt = blockIdx.x % KT;
    const int h = (blockIdx.x / KT) % p.H;
    const int b = blockIdx.x / (KT * p.H);
    int map, krow;
    kv_tile(p, kt, map, krow);
    const int T = p.q_tiles;

    if (warp == 4) {
        if (lane == 0) {
            mbar_arrive_expect_tx(sh.stat_full, 2 * TILE);
            for (int half = 0; half < 2; half++) {
                tma_load_4d(smem + SMEM_STAT + half * PANEL, map ? &tm_jk : &tm_k, sh.stat_full, half * 64, h, krow,
                            b);
                tma_load_4d(smem + SMEM_STAT + TILE + half * PANEL, map ? &tm_jv : &tm_v, sh.stat_full, half * 64,
                            h, krow, b);
            }
            int issued = 0;
            for (int t = 0; t < T; t++) {
                const int slot = t & 1;
                if (!mbar_wait(&sh.ld_empty[slot], ((t >> 1) & 1) ^ 1, w)) break;
                mbar_arrive_expect_tx(&sh.ld_full[slot], 2 * TILE);
                uint8_t *dst = smem + SMEM_RING + slot * 2 * TILE;
                for (int half = 0; half < 2; half++) {
                    tma_load_4d(dst + half * PANEL, &tm_q, &sh.ld_full[slot], half * 64, h, t * BM, b);
                    tma_load_4d(dst + TILE + half * PANEL, &tm_do, &sh.ld_full[slot], half * 64, h, t * BM, b);
                }
                issued++;
            }
            mbar_drain(sh.stat_full, 0, DRAIN_NS);
            for (int t = issued > 2 ? issued - 2 : 0; t < issued; t++)
                mbar_drain(&sh.ld_full[t & 1], (t >> 1) & 1, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t tS = tmem, tP = tmem + 128, tV = tmem + 256, tK = tmem + 384;
            const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + SMEM_STAT), 16, 1024);      // K (K-major)
            const uint64_t dv0 = dk0 + (uint64_t)(TILE >> 4);                             // V (K-major)
            const uint64_t dring = smem_desc_sw128(smem_u32(smem + SMEM_RING), 16, 1024);  // Q / dO (K-major)
            const uint64_t dring_mn = smem_desc_sw128(smem_u32(smem + SMEM_RING), PANEL, 1024);
            bool ok = mbar_wait(sh.stat_full, 0, w);
            for (int t = 0; t < T && ok; t++) {
                const int slot = t & 1;
                if (!(ok = mbar_wait(&sh.ld_full[slot], (t >> 1) & 1, w))) break;
                tc_fence_after();
                const uint64_t qdesc = dring + (uint64_t)((slot * 2 * TILE) >> 4);
                const uint64_t odesc = qdesc + (uint64_t)(TILE >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    const uint64_t off = (uint64_t)((kk >> 2) * PANEL + (kk & 3) * 32) >> 4;
                    mma_ss(tS, dk0 + off, qdesc + off, p.idesc_qk, kk > 0);     // S^T = K Q^T
                    mma_ss(tP, dv0 + off, odesc + off, p.idesc_bf16, kk > 0);   // dP^T = V dO^T
                }
                tc_commit(sh.s_full);
                if (!(ok = mbar_wait(sh.ds_full, t & 1, w))) break;
                tc_fence_after();
                const uint64_t qmn = dring_mn + (uint64_t)((slot * 2 * TILE) >> 4);
                const uint64_t omn = qmn + (uint64_t)(TILE >> 4);
#pragma unroll
                for (int kk = 0; kk < BM / 16; kk++) {
                    const uint64_t off = (uint64_t)((kk * 16 * 128) >> 4);
                    mma_ts(tV, tS + kk * 8, omn + off, p.idesc_bf16 | (1u << 16), (t > 0 || kk > 0) ? 1u : 0u);
                    mma_ts(tK, tP + kk * 8, qmn + off, p.idesc_ds_q, (t > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&sh.ld_empty[slot]);
            }
            tc_commit(sh.acc_done);
            tc_commit(sh.drain);
            mbar_drain(sh.drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ compute: one key row per thread
        const int r = threadIdx.x;
        const uint32_t lb = tmem + ((uint32_t)(32 * warp) << 16);
        const float sl2 = p.scale_log2;
        const float *lse_bh = p.lse + ((long)b * p.H + h) * p.S;
        const float *d_bh = p.Dsum + ((long)b * p.H + h) * p.S;
        bool ok = true;
        for (int t = 0; t < T; t++) {
            if (!mbar_wait(sh.s_full, t & 1, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t sv[32], pv[32], pk[16], ds[16];
                tmem_ld32(lb + c * 32, sv);
                tmem_ld32(lb + 128 + c * 32, pv);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    float pe[2], de[2];
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const long qrow = (long)t * BM + c * 32 + k + e;  // column = query row (warp-uniform)
                        if (qrow < p.S) {
                            const float l2 = __ldg(lse_bh + qrow) * 1.4426950408889634f;
                            pe[e] = ex2(fmaf(__uint_as_float(sv[k + e]), sl2, -l2));
                            de[e] = pe[e] * (__uint_as_float(pv[k + e]) - __ldg(d_bh + qrow));
                        } else {
                            pe[e] = 0.f;
                            de[e] = 0.f;
                        }
                    }
                    pk[k / 2] = pack_bf16x2(pe[0], pe[1]);
                    ds[k / 2] = pack2(de[0], de[1], p.ds_f16);
                }
                tmem_st16(lb + c * 16, pk);        // P^T over S^T
                tmem_st16(lb + 128 + c * 16, ds);  // dS^T over dP^T
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(sh.ds_full);
        }
        if (ok && mbar_wait(sh.acc_done, 0, w)) {
            tc_fence_after();
            const long kr = (long)krow + r;
            const long rows = map ? p.Nj : p.Nv;
            const bool live = kr < rows;
            const long off = (((long)b * rows + (live ? kr : 0)) * p.H + h) * D;
            float *dkp = (map ? p.djk : p.dk) + off;
            float *dvp = (map ? p.djv : p.dv) + off;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t gk[32], gv[32];
                tmem_ld32(lb + 384 + c * 32, gk);
                tmem_ld32(lb + 256 + c * 32, gv);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        *reinterpret_cast<float4 *>(dkp + c * 32 + k) =
                            make_float4(__uint_as_float(gk[k]) * p.scale, __uint_as_float(gk[k + 1]) * p.scale,
                                        __uint_as_float(gk[k + 2]) * p.scale, __uint_as_float(gk[k + 3]) * p.scale);
                        *reinterpret_cast<float4 *>(dvp + c * 32 + k) =
                            make_float4(__uint_as_float(gv[k]), __uint_as_float(gv[k + 1]), __uint_as_float(gv[k + 2]),
                                        __uint_as_float(gv[k + 3]));
                    }
                }
            }
        }
    }
    bw_teardown(tmem);
}

// ------------------------------------------------------------------- host

static bool bw_map(CUtensorMap *m, const void *base, long rows, int H, int B, bool f16, const char **why) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [&] {
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode) {
        if (why) *why = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    cuuint64_t dims[4] = {(cuuint64_t)bw::D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)bw::D * 2, (cuuint64_t)H * bw::D * 2, (cuuint64_t)rows * H * bw::D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)bw::BM, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled rejected a tensor";
        return false;
    }
    return true;
}

cudaError_t launch_attn_bwd(const Geom &g, bool qk_f16, const void *q, const void *k, const void *v, const void *jk,
                            const void *jv, const void *out, const void *dout, const float *lse, float *Dsum, float *dq,
                            float *dk, float *dv, float *djk, float *djv, unsigned long long wait_limit_ns, int *err,
                            cudaStream_t st, const char **why) {
    const long rows = (long)g.B * g.S * g.H;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    bwd_dsum_kernel<<<(unsigned)sms * 8, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(out),
                                                       static_cast<const __nv_bfloat16 *>(dout), g.S, g.H, g.B, Dsum);
    CUtensorMap mq, mdo, mk, mv, mjk, mjv;
    const bool has_joint = g.Nj > 0;
    if (!bw_map(&mq, q, g.S, g.H, g.B, qk_f16, why) || !bw_map(&mdo, dout, g.S, g.H, g.B, false, why) ||
        !bw_map(&mk, k, g.Nv, g.H, g.B, qk_f16, why) || !bw_map(&mv, v, g.Nv, g.H, g.B, false, why) ||
        !bw_map(&mjk, has_joint ? jk : k, has_joint ? g.Nj : g.Nv, g.H, g.B, qk_f16, why) ||
        !bw_map(&mjv, has_joint ? jv : v, has_joint ? g.Nj : g.Nv, g.H, g.B, false, why))
        return cudaErrorInvalidValue;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bw::SMEM_ALLOC);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            bw::SMEM_ALLOC);
    });
    if (attr_err != cudaSuccess) return attr_err;
    BwParams p;
    p.S = g.S, p.Nv = g.Nv, p.Nj = g.Nj, p.H = g.H;
    p.q_tiles = (int)((g.S + bw::BM - 1) / bw::BM);
    p.kv_tiles_v = (int)((g.Nv + bw::BM - 1) / bw::BM);
    p.kv_tiles_j = (int)((g.Nj + bw::BM - 1) / bw::BM);
    p.scale = (float)(1.0 / sqrt((double)g.d));
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
    p.lse = lse, p.Dsum = Dsum;
    p.dq = dq, p.dk = dk, p.dv = dv, p.djk = djk, p.djv = djv;
    // A/B formats: bits 7-9 and 10-12 (0 = fp16, 1 = bf16); bit 16: B MN-major
    const uint32_t base = idesc_bf16_f32(bw::BM, bw::BM, false) & ~((7u << 7) | (7u << 10));
    const uint32_t f16 = base, bf16 = base | (1u << 7) | (1u << 10);
    p.idesc_qk = qk_f16 ? f16 : bf16;          // S = Q K^T
    p.idesc_bf16 = bf16;                       // dP = dO V^T (and dV with the MN bit)
    p.idesc_ds_k = (qk_f16 ? f16 : bf16) | (1u << 16);  // dQ += dS K  (dS in K's type, K MN-major)
    p.idesc_ds_q = (qk_f16 ? f16 : bf16) | (1u << 16);  // dK += dS^T Q
    p.ds_f16 = qk_f16 ? 1 : 0;
    p.wait_limit_ns = wait_limit_ns;
    p.err = err;
    const long dq_grid = (long)g.B * g.H * p.q_tiles;
    const long dkv_grid = (long)g.B * g.H * (p.kv_tiles_v + p.kv_tiles_j);
    bwd_dq_kernel<<<(unsigned)dq_grid, bw::THREADS, bw::SMEM_ALLOC, st>>>(mq, mdo, mk, mv, mjk, mjv, p);
    bwd_dkv_kernel<<<(unsigned)dkv_grid, bw::THREADS, bw::SMEM_ALLOC, st>>>(mq, mdo, mk, mv, mjk, mjv, p);
    return cudaGetLastError();
}

}  // namespace k6
