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
// operand streamed by TMA.  Warps 0-7 form P/dS (two warpgroups, each owning
// half of a tile's columns; one TMEM lane = one row per thread), warp 8 drives
// TMA, warp 9 owns tensor memory and one of its threads issues every MMA.
//
//   dq kernel  (Q, dO stationary; K through a 3-slot ring, V through 2 slots):
//     S = Q K_j^T, dP = dO V_j^T (SS) into columns 0-127 / 128-255; dS (q/k
//     type) goes to one of two spare buffers (384-447, 448-511), so the MMAs
//     of tile j+1 start before dQ += dS_j K_j (TS, 256-383) and that product
//     runs under the next tile's row pass.
//   dkv kernel (K, V stationary; Q/dO through a 2-slot ring):
//     S^T = K Q_i^T, dP^T = V dO_i^T (SS) into 0-127 / 128-255; P^T goes to
//     shared memory (K-major, 128-byte swizzle) and dS^T over dP^T, so
//     S^T of tile i+1 runs under the row pass of tile i; then
//     dV += P^T dO_i (SS) and dK += dS^T Q_i (TS) into 256-383 / 384-511.
// MMAs of one thread run in issue order, so an MMA may overwrite tensor
// memory that an earlier MMA reads (dP of tile i+1 over dS^T of tile i).
// All waits are bounded like the forward kernel's.  Gradients are fp32.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>


#include "k6_device.cuh"
#include "k6_internal.h"

namespace k6 {

namespace bw {
constexpr int D = 128, BM = 128;
constexpr int PANEL = BM * 64 * 2;          // 128 rows x 64 elements of 16 bits
constexpr int TILE = 2 * PANEL;             // 32 KB: 128 rows x 128 elements
constexpr int THREADS = 320;                // warps 0-7 rows, 8 TMA, 9 MMA + TMEM
constexpr int SMEM_DATA = 7 * TILE;         // both kernels: 224 KB of tiles
constexpr int SMEM_ALLOC = SMEM_DATA + 256 + 1024;  // barriers, TMEM slot, abort flag, alignment
constexpr unsigned long long DRAIN_NS = 1000000000ull;
constexpr float LOG2E = 1.4426950408889634f;
}  // namespace bw

struct BwParams {
    long S, Nv, Nj;
    int H, q_tiles, kv_tiles_v, kv_tiles_j;
    float scale_log2, scale;                // log2(e)/sqrt(d), 1/sqrt(d)
    const float2 *LD;                       // [B][H][S] {lse * log2(e), D}
    float *dq, *dk, *dv, *djk, *djv;        // fp32 gradients
    uint32_t idesc_qk, idesc_bf16, idesc_bf16_mn, idesc_ds_mn;
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

// 32 lanes x 16 consecutive 32-bit columns (load) / 8 columns (store).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// 2^x on the special function unit, kept in program order (volatile) so the
// exps of a row pass run before the wait that follows them.
__device__ __forceinline__ float ex2_here(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ------------------------------------------------------------- pre-pass D

// LD[(b*H + h)*S + s] = {lse * log2(e), sum_e dout * out} for one head row.
// Half a warp (16 lanes x 8 elements) covers one d = 128 row.
__global__ void __launch_bounds__(256) bwd_dsum_kernel(const __nv_bfloat16 *__restrict__ out,
                                                      const __nv_bfloat16 *__restrict__ dout,
                                                      const float *__restrict__ lse, long S, int H, int B,
                                                      float2 *__restrict__ LD) {
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
            const long li = ((bs / S) * H + h) * S + bs % S;
            LD[li] = make_float2(lse[li] * bw::LOG2E, s);
        }
    }
}

// ----------------------------------------------------------- shared set-up

// Barriers 0..NB-1 with the given arrival counts, 512 TMEM columns (warp 9).
template <int NB>
__device__ __forceinline__ uint32_t bw_setup(uint8_t *smem, const int (&counts)[NB], uint64_t *&bars,
                                             volatile int *&abort_flag) {
    bars = reinterpret_cast<uint64_t *>(smem + bw::SMEM_DATA);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NB);
    abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NB; i++) mbar_init(bars + i, counts[i]);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x / 32 == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *tmem_slot;
}

__device__ __forceinline__ void bw_teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x / 32 == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Key tile t of concat(k, joint_k): which map (0 video, 1 joint) and first row.
__device__ __forceinline__ void kv_tile(const BwParams &p, int t, int &map, int &row) {
    if (t < p.kv_tiles_v) {
        map = 0;
        row = t * bw::BM;
    } else {
        map = 1;
        row = (t - p.kv_tiles_v) * bw::BM;
    }
}

// Two 64-element panels of a 128-row tile into dst (32 KB, completes on bar).
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *m, uint64_t *bar, int h, int row, int b) {
    tma_load_4d(dst, m, bar, 0, h, row, b);
    tma_load_4d(dst + bw::PANEL, m, bar, 64, h, row, b);
}

// Step kk of a K-major SS MMA chain over d = 128 (both operands 128-byte swizzled),
// issued by the elected lane of the converged calling warp.
__device__ __forceinline__ void mma_kmajor(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int kk) {
    const uint64_t off = (uint64_t)((kk >> 2) * bw::PANEL + (kk & 3) * 32) >> 4;
    mma_ss_w(d, a + off, b + off, idesc, kk > 0);
}

// Epilogue: 64 fp32 columns of this thread's TMEM lane, times `scale`, to dst.
__device__ __forceinline__ void store_row64(uint32_t taddr, float *dst, float scale, bool live) {
#pragma unroll
    for (int c = 0; c < 2; c++) {
        uint32_t o[32];
        tmem_ld32(taddr + c * 32, o);
        tmem_ld_wait();
        if (live) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4 *>(dst + c * 32 + k) =
                    make_float4(__uint_as_float(o[k]) * scale, __uint_as_float(o[k + 1]) * scale,
                                __uint_as_float(o[k + 2]) * scale, __uint_as_float(o[k + 3]) * scale);
        }
    }
}

// ------------------------------------------------------------------ dq kernel
//
// smem tiles: Q 0, dO 1, K slots 2-4, V slots 5-6.
// barriers: stat_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full,
//           ds_full (256 arrivals), acc_done, drain.

namespace dqb {
constexpr int STAT = 0, KFULL = 1, KEMPTY = 4, VFULL = 7, VEMPTY = 9, SFULL = 11, DSFULL = 12, ACC = 13,
              DRAIN = 14, NB = 15;
}

__global__ void __launch_bounds__(bw::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_jk, const __grid_constant__ CUtensorMap tm_jv,
                  const BwParams p) {
    using namespace bw;
    using namespace dqb;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int counts[NB] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 256, 1, 1};
    uint64_t *bar;
    volatile int *abort_flag;
    const uint32_t tmem = bw_setup<NB>(smem, counts, bar, abort_flag);
    const WaitCtx w{p.wait_limit_ns, p.err, abort_flag};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = blockIdx.x % p.q_tiles;
    const int h = (blockIdx.x / p.q_tiles) % p.H;
    const int b = blockIdx.x / (p.q_tiles * p.H);
    const int q0 = qt * BM;
    const int T = p.kv_tiles_v + p.kv_tiles_j;
    uint8_t *sQ = smem, *sDO = smem + TILE, *sK = smem + 2 * TILE, *sV = smem + 5 * TILE;

    // The control warps run whole and converged: every lane waits (a warp-uniform
    // vote), one elected lane arms barriers, issues copies, MMAs and commits.
    if (warp == 8) {
        {
            const bool leader = elect_one();
            if (leader) {
                mbar_arrive_expect_tx(bar + STAT, 2 * TILE);
                load_tile(sQ, &tm_q, bar + STAT, h, q0, b);
                load_tile(sDO, &tm_do, bar + STAT, h, q0, b);
            }
            int nk = 0, nv = 0;  // K and V tiles issued
            for (int t = 0; t < T; t++) {
                const int ks = t % 3, vs = t & 1;
                int map, row;
                kv_tile(p, t, map, row);
                if (!mbar_wait_w(bar + KEMPTY + ks, ((t / 3) & 1) ^ 1, w)) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar + KFULL + ks, TILE);
                    load_tile(sK + ks * TILE, map ? &tm_jk : &tm_k, bar + KFULL + ks, h, row, b);
                }
                nk++;
                if (!mbar_wait_w(bar + VEMPTY + vs, ((t >> 1) & 1) ^ 1, w)) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar + VFULL + vs, TILE);
                    load_tile(sV + vs * TILE, map ? &tm_jv : &tm_v, bar + VFULL + vs, h, row, b);
                }
                nv++;
            }
            // let copies in flight land before the CTA exits
            mbar_drain(bar + STAT, 0, DRAIN_NS);
            for (int t = nk > 3 ? nk - 3 : 0; t < nk; t++) mbar_drain(bar + KFULL + t % 3, (t / 3) & 1, DRAIN_NS);
            for (int t = nv > 2 ? nv - 2 : 0; t < nv; t++) mbar_drain(bar + VFULL + (t & 1), (t >> 1) & 1, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp == 9) {
        {
            const uint32_t tS = tmem, tP = tmem + 128, tA = tmem + 256, tDS = tmem + 384;
            const uint64_t dq_ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t ddo = smem_desc_sw128(smem_u32(sDO), 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), 16, 1024);
            const uint64_t dkmn = smem_desc_sw128(smem_u32(sK), PANEL, 1024);
            // S(t) = Q K^T and dP(t) = dO V^T, two interleaved chains; then free the
            // V slot and publish S/dP (each commit also covers every earlier MMA).
            auto issue_sdp = [&](int t) -> bool {
                const int ks = t % 3, vs = t & 1;
                if (!mbar_wait_w(bar + KFULL + ks, (t / 3) & 1, w)) return false;
                if (!mbar_wait_w(bar + VFULL + vs, (t >> 1) & 1, w)) return false;
                tc_fence_after();
                const uint64_t kd = dk0 + (uint64_t)((ks * TILE) >> 4), vd = dv0 + (uint64_t)((vs * TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    mma_kmajor(tS, dq_, kd, p.idesc_qk, kk);
                    mma_kmajor(tP, ddo, vd, p.idesc_bf16, kk);
                }
                tc_commit_w(bar + VEMPTY + vs);
                tc_commit_w(bar + SFULL);
                return true;
            };
            bool ok = mbar_wait_w(bar + STAT, 0, w) && T > 0 && issue_sdp(0);
            for (int t = 0; t < T && ok; t++) {
                // the row pass has read S(t)/dP(t) and written dS(t) to buffer t & 1
                if (!(ok = mbar_wait_w(bar + DSFULL, t & 1, w))) break;
                tc_fence_after();
                if (t + 1 < T && !(ok = issue_sdp(t + 1))) break;
                const uint64_t kmn = dkmn + (uint64_t)(((t % 3) * TILE) >> 4);
                const uint32_t ads = tDS + (t & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < BM / 16; kk++)
                    mma_ts_w(tA, ads + kk * 8, kmn + (uint64_t)((kk * 16 * 128) >> 4), p.idesc_ds_mn,
                           (t > 0 || kk > 0) ? 1u : 0u);  // dQ += dS K
                tc_commit_w(bar + KEMPTY + t % 3);
            }
            if (ok) tc_commit_w(bar + ACC);
            tc_commit_w(bar + DRAIN);
            mbar_drain(bar + DRAIN, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        // ------------------------------------------ rows: lane quarter q4, key half g
        const int q4 = warp & 3, g = warp >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lb = tmem + ((uint32_t)(32 * q4) << 16);
        const long grow = (long)q0 + r;
        const bool live = grow < p.S;
        const float2 ld = live ? p.LD[((long)b * p.H + h) * p.S + grow] : make_float2(0.f, 0.f);
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int t = 0; t < T; t++) {
            if (!mbar_wait(bar + SFULL, t & 1, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; c++) {
                uint32_t sv[32], pv[32], ds[16];
                tmem_ld32(lb + 64 * g + 32 * c, sv);
                tmem_ld32(lb + 128 + 64 * g + 32 * c, pv);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const float p0 = ex2(fmaf(__uint_as_float(sv[k]), sl2, -ld.x));
                    const float p1 = ex2(fmaf(__uint_as_float(sv[k + 1]), sl2, -ld.x));
                    ds[k / 2] = pack2(p0 * (__uint_as_float(pv[k]) - ld.y), p1 * (__uint_as_float(pv[k + 1]) - ld.y),
                                      p.ds_f16);
                }
                tmem_st16(lb + 384 + 64 * (t & 1) + 32 * g + 16 * c, ds);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar + DSFULL);
        }
        if (ok && mbar_wait(bar + ACC, 0, w)) {
            tc_fence_after();
            store_row64(lb + 256 + 64 * g, p.dq + (((long)b * p.S + (live ? grow : 0)) * p.H + h) * D + 64 * g,
                        p.scale, live);
        }
    }
    bw_teardown(tmem);
}

// Row pass of the dk/dv kernel for one key row and 64 queries (FULL: all live).
// P for the 64 queries from S^T in registers; queries j >= nq get P = 0.
template <bool FULL>
__device__ __forceinline__ void p_half(float (&pr)[64], const uint32_t (&sv)[2][32], const float2 *ldq, int nq,
                                       float sl2) {
#pragma unroll
    for (int c = 0; c < 2; c++) {
#pragma unroll
        for (int k = 0; k < 32; k++) {
            const int j = 32 * c + k;
            const float l2 = (FULL || j < nq) ? ldq[j].x : __int_as_float(0x7f800000);
            pr[j] = ex2_here(fmaf(__uint_as_float(sv[c][k]), sl2, -l2));
        }
        asm volatile("" ::: "memory");  // one half's loads at a time (register pressure)
    }
}

// dS^T = P (dP^T - D) over 16-query chunks [C0, C1) of the 64 columns at taddr
// (each chunk's dS^T lands on columns already read), and P rounded to bf16 into
// this thread's row of the swizzled P^T panel at prow.
template <bool FULL, int C0, int C1>
__device__ __forceinline__ void ds_half(const float (&pr)[64], const float2 *ldq, int nq, uint32_t taddr,
                                        uint32_t prow, int r, int ds_f16) {
#pragma unroll
    for (int c = C0; c < C1; c++) {
        uint32_t pv[16], ds[8], pk[8];
        tmem_ld16(taddr + 16 * c, pv);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            float de[2];
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int j = 16 * c + k + e;
                // plain load: the clobber of the tensor-memory load above keeps it in this chunk
                const float dd = (FULL || j < nq) ? ldq[j].y : 0.f;
                de[e] = pr[j] * (__uint_as_float(pv[k + e]) - dd);
            }
            ds[k / 2] = pack2(de[0], de[1], ds_f16);
            pk[k / 2] = pack_bf16x2(pr[16 * c + k], pr[16 * c + k + 1]);
        }
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int chunk = 2 * c + i;  // 16-byte chunk of the 128-byte row
            st_shared_v4(prow + ((chunk ^ (r & 7)) << 4), pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        tmem_st8(taddr + 8 * c, ds);
    }
}

// ----------------------------------------------------------------- dkv kernel
//
// smem tiles: K 0, V 1, ring slot s: Q 2+2s, dO 3+2s; P^T 6.
// barriers: stat_full, q_full[2], do_full[2], q_empty[2], do_empty[2], s_ready
//           (S^T(i) done), consumed (256 arrivals: S^T(i) read), pds_ready[2] (256
//           arrivals each: P^T(i) in shared memory and dS^T(i) in tensor memory for
//           the first / last 32 queries of each half), window (dV/dK(i-1) and
//           dP^T(i) done), acc_done, drain.
// Q and dO slots are released separately: Q(i) once dK(i) is done, midway
// through the window, so Q(i+2) is in flight while the window finishes.
//
// Per tile i the MMA thread issues S^T(i+1) as soon as the row pass has read
// S^T(i).  The row pass publishes P^T(i)/dS^T(i) in two parts (queries 0-31 and
// 64-95, then 32-63 and 96-127: the first half of each warpgroup's columns), so
// the window starts on the first part while the second is formed: dK(i) | dV(i)
// over the first part's 4 K-steps, then over the second part's (dK) and two of
// dV's, then dP^T(i+1) | the last two dV steps (dP^T(i+1) overwrites dS^T(i),
// so it follows every dK(i) MMA).  The row pass of tile i+1 computes its P from
// S^T(i+1) while that window runs, and only the dS / P^T stores wait for it.

namespace dkvb {
constexpr int STAT = 0, QFULL = 1, DOFULL = 3, QEMPTY = 5, DOEMPTY = 7, SREADY = 9, CONSUMED = 10, PDS = 11,
              WIN = 13, ACC = 14, DRAIN = 15, NB = 16;  // PDS, PDS + 1: the two parts of a tile's P^T / dS^T
}

__global__ void __launch_bounds__(bw::THREADS, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_jk, const __grid_constant__ CUtensorMap tm_jv,
                   const BwParams p) {
    using namespace bw;
    using namespace dkvb;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int counts[NB] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 256, 256, 256, 1, 1, 1};
    uint64_t *bar;
    volatile int *abort_flag;
    const uint32_t tmem = bw_setup<NB>(smem, counts, bar, abort_flag);
    const WaitCtx w{p.wait_limit_ns, p.err, abort_flag};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int KT = p.kv_tiles_v + p.kv_tiles_j;
    const int kt = blockIdx.x % KT;
    const int h = (blockIdx.x / KT) % p.H;
    const int b = blockIdx.x / (KT * p.H);
    int map, krow;
    kv_tile(p, kt, map, krow);
    const int T = p.q_tiles;
    uint8_t *sK = smem, *sV = smem + TILE, *sRing = smem + 2 * TILE, *sP = smem + 6 * TILE;

    // The control warps run whole and converged: every lane waits (a warp-uniform
    // vote), one elected lane arms barriers, issues copies, MMAs and commits.
    if (warp == 8) {
        {
            const bool leader = elect_one();
            if (leader) {
                mbar_arrive_expect_tx(bar + STAT, 2 * TILE);
                load_tile(sK, map ? &tm_jk : &tm_k, bar + STAT, h, krow, b);
                load_tile(sV, map ? &tm_jv : &tm_v, bar + STAT, h, krow, b);
            }
            int nq = 0, ndo = 0;  // Q and dO tiles issued
            for (int t = 0; t < T; t++) {
                const int s = t & 1;
                const uint32_t par = ((t >> 1) & 1) ^ 1;
                if (!mbar_wait_w(bar + QEMPTY + s, par, w)) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar + QFULL + s, TILE);
                    load_tile(sRing + 2 * s * TILE, &tm_q, bar + QFULL + s, h, t * BM, b);
                }
                nq++;
                if (!mbar_wait_w(bar + DOEMPTY + s, par, w)) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar + DOFULL + s, TILE);
                    load_tile(sRing + (2 * s + 1) * TILE, &tm_do, bar + DOFULL + s, h, t * BM, b);
                }
                ndo++;
            }
            mbar_drain(bar + STAT, 0, DRAIN_NS);
            for (int t = nq > 2 ? nq - 2 : 0; t < nq; t++) mbar_drain(bar + QFULL + (t & 1), (t >> 1) & 1, DRAIN_NS);
            for (int t = ndo > 2 ? ndo - 2 : 0; t < ndo; t++)
                mbar_drain(bar + DOFULL + (t & 1), (t >> 1) & 1, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp == 9) {
        {
            const uint32_t tS = tmem, tP = tmem + 128, tV = tmem + 256, tK = tmem + 384;
            const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), 16, 1024);
            const uint64_t dring = smem_desc_sw128(smem_u32(sRing), 16, 1024);
            const uint64_t dring_mn = smem_desc_sw128(smem_u32(sRing), PANEL, 1024);
            const uint64_t dp = smem_desc_sw128(smem_u32(sP), 16, 1024);
            // descriptor of tile `which` (0 Q, 1 dO) of the ring slot of tile t
            auto slot = [&](uint64_t base, int t, int which) {
                return base + (uint64_t)(((2 * (t & 1) + which) * TILE) >> 4);
            };
            auto wait_q = [&](int t) { return mbar_wait_w(bar + QFULL + (t & 1), (t >> 1) & 1, w); };
            auto wait_do = [&](int t) { return mbar_wait_w(bar + DOFULL + (t & 1), (t >> 1) & 1, w); };
            bool ok = mbar_wait_w(bar + STAT, 0, w) && T > 0 && wait_q(0);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) mma_kmajor(tS, dk0, slot(dring, 0, 0), p.idesc_qk, kk);  // S^T = K Q^T
                tc_commit_w(bar + SREADY);
                ok = wait_do(0);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) mma_kmajor(tP, dv0, slot(dring, 0, 1), p.idesc_bf16, kk);  // dP^T = V dO^T
                tc_commit_w(bar + WIN);
            }
            for (int t = 0; t < T && ok; t++) {
                // the row pass has read S^T(t): S^T(t+1) may overwrite its columns
                if (!(ok = mbar_wait_w(bar + CONSUMED, t & 1, w))) break;
                tc_fence_after();
                const bool next = t + 1 < T;
                if (next) {
                    if (!(ok = wait_q(t + 1))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++) mma_kmajor(tS, dk0, slot(dring, t + 1, 0), p.idesc_qk, kk);
                    tc_commit_w(bar + SREADY);
                }
                // the first part of P^T(t) is in shared memory and of dS^T(t) over dP^T(t)
                if (!(ok = mbar_wait_w(bar + PDS, t & 1, w))) break;
                if (next && !(ok = wait_do(t + 1))) break;
                tc_fence_after();
                const uint32_t acc = t > 0 ? 1u : 0u;
                // K-step kk covers queries 16 kk .. 16 kk + 15: the first part holds kk 0, 1, 4, 5
                auto dv_step = [&](int kk) {  // dV += P^T dO
                    const uint64_t poff = (uint64_t)((kk >> 2) * PANEL + (kk & 3) * 32) >> 4;
                    mma_ss_w(tV, dp + poff, slot(dring_mn, t, 1) + (uint64_t)((kk * 16 * 128) >> 4), p.idesc_bf16_mn,
                           acc | (kk > 0 ? 1u : 0u));
                };
                auto dk_step = [&](int kk) {  // dK += dS^T Q
                    mma_ts_w(tK, tP + (kk >> 2) * 64 + (kk & 3) * 8,
                           slot(dring_mn, t, 0) + (uint64_t)((kk * 16 * 128) >> 4), p.idesc_ds_mn,
                           acc | (kk > 0 ? 1u : 0u));
                };
                constexpr int part0[4] = {0, 1, 4, 5}, part1[4] = {2, 3, 6, 7};
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    dk_step(part0[i]);
                    dv_step(part0[i]);
                }
                if (!(ok = mbar_wait_w(bar + PDS + 1, t & 1, w))) break;
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    dk_step(part1[i]);
                    if (i < 2) dv_step(part1[i]);
                }
                tc_commit_w(bar + QEMPTY + (t & 1));  // Q(t): S^T(t) and dK(t) done
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    if (next) mma_kmajor(tP, dv0, slot(dring, t + 1, 1), p.idesc_bf16, kk);  // dP^T(t+1)
                    if (kk < 2) dv_step(part1[2 + kk]);
                }
                tc_commit_w(bar + DOEMPTY + (t & 1));  // dO(t): dP^T(t) and dV(t) done
                tc_commit_w(bar + WIN);
            }
            if (ok) tc_commit_w(bar + ACC);
            tc_commit_w(bar + DRAIN);
            mbar_drain(bar + DRAIN, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        // ------------------------------------------ rows: key row r, query half g
        const int q4 = warp & 3, g = warp >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lb = tmem + ((uint32_t)(32 * q4) << 16);
        const float sl2 = p.scale_log2;
        const float2 *ld_bh = p.LD + ((long)b * p.H + h) * p.S;
        // this thread's row of P^T panel g: 8 chunks of 16 bytes, 128-byte swizzle
        const uint32_t prow = smem_u32(sP) + g * PANEL + (r >> 3) * 1024 + (r & 7) * 128;
        bool ok = true;
        for (int t = 0; t < T; t++) {
            if (!mbar_wait(bar + SREADY, t & 1, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // S^T of this half into registers, then its columns are free for S^T(t+1)
            uint32_t sv[2][32];
            tmem_ld32(lb + 64 * g, sv[0]);
            tmem_ld32(lb + 64 * g + 32, sv[1]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bar + CONSUMED);
            // P = 2^(s log2(e)/sqrt(d) - lse log2(e)); queries past S get lse = +inf, so P = 0
            const long qb = (long)t * BM + 64 * g;  // first query of this half
            const float2 *ldq = ld_bh + qb;
            const int nq = p.S - qb >= 64 ? 64 : (int)(p.S - qb);  // live queries of this half (warp-uniform)
            float pr[64];
            if (nq == 64)
                p_half<true>(pr, sv, ldq, 64, sl2);
            else
                p_half<false>(pr, sv, ldq, nq, sl2);
            // dV/dK(t-1) and dP^T(t) done: the P^T buffer is free and dP^T(t) is in place
            if (!mbar_wait(bar + WIN, t & 1, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // first part (queries 0-31 of this half), published before the second is formed
            if (nq == 64)
                ds_half<true, 0, 2>(pr, ldq, 64, lb + 128 + 64 * g, prow, r, p.ds_f16);
            else
                ds_half<false, 0, 2>(pr, ldq, nq, lb + 128 + 64 * g, prow, r, p.ds_f16);
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar + PDS);
            if (nq == 64)
                ds_half<true, 2, 4>(pr, ldq, 64, lb + 128 + 64 * g, prow, r, p.ds_f16);
            else
                ds_half<false, 2, 4>(pr, ldq, nq, lb + 128 + 64 * g, prow, r, p.ds_f16);
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar + PDS + 1);
        }
        if (ok && mbar_wait(bar + ACC, 0, w)) {
            tc_fence_after();
            const long kr = (long)krow + r;
            const long rows = map ? p.Nj : p.Nv;
            const bool live = kr < rows;
            const long off = (((long)b * rows + (live ? kr : 0)) * p.H + h) * D + 64 * g;
            store_row64(lb + 384 + 64 * g, (map ? p.djk : p.dk) + off, p.scale, live);
            store_row64(lb + 256 + 64 * g, (map ? p.djv : p.dv) + off, 1.0f, live);
        }
    }
    bw_teardown(tmem);
}

// ------------------------------------------------------------------- host

cudaError_t launch_attn_bwd(const Geom &g, bool qk_f16, const void *q, const void *k, const void *v, const void *jk,
                            const void *jv, const void *out, const void *dout, const float *lse, float2 *LD, float *dq,
                            float *dk, float *dv, float *djk, float *djv, unsigned long long wait_limit_ns, int *err,
                            cudaStream_t st, const char **why) {
    const long rows = (long)g.B * g.S * g.H;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    CUtensorMap mq, mdo, mk, mv, mjk, mjv;
    const bool has_joint = g.Nj > 0;
    if (!make_bshd_map(&mq, q, g.S, g.H, g.B, qk_f16, why) || !make_bshd_map(&mdo, dout, g.S, g.H, g.B, false, why) ||
        !make_bshd_map(&mk, k, g.Nv, g.H, g.B, qk_f16, why) || !make_bshd_map(&mv, v, g.Nv, g.H, g.B, false, why) ||
        !make_bshd_map(&mjk, has_joint ? jk : k, has_joint ? g.Nj : g.Nv, g.H, g.B, qk_f16, why) ||
        !make_bshd_map(&mjv, has_joint ? jv : v, has_joint ? g.Nj : g.Nv, g.H, g.B, false, why))
        return cudaErrorInvalidValue;
    cudaError_t attr_err = set_max_dynamic_smem((const void *)bwd_dq_kernel, bw::SMEM_ALLOC);
    if (attr_err == cudaSuccess) attr_err = set_max_dynamic_smem((const void *)bwd_dkv_kernel, bw::SMEM_ALLOC);
    if (attr_err != cudaSuccess) return attr_err;
    bwd_dsum_kernel<<<(unsigned)sms * 8, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(out),
                                                       static_cast<const __nv_bfloat16 *>(dout), lse, g.S, g.H, g.B,
                                                       LD);
    BwParams p;
    p.S = g.S, p.Nv = g.Nv, p.Nj = g.Nj, p.H = g.H;
    p.q_tiles = (int)((g.S + bw::BM - 1) / bw::BM);
    p.kv_tiles_v = (int)((g.Nv + bw::BM - 1) / bw::BM);
    p.kv_tiles_j = (int)((g.Nj + bw::BM - 1) / bw::BM);
    p.scale = (float)(1.0 / sqrt((double)g.d));
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
    p.LD = LD;
    p.dq = dq, p.dk = dk, p.dv = dv, p.djk = djk, p.djv = djv;
    // A/B formats: bits 7-9 and 10-12 (0 = fp16, 1 = bf16); bit 16: B MN-major
    const uint32_t base = idesc_bf16_f32(bw::BM, bw::BM, false) & ~((7u << 7) | (7u << 10));
    const uint32_t f16 = base, bf16 = base | (1u << 7) | (1u << 10);
    p.idesc_qk = qk_f16 ? f16 : bf16;                    // S = Q K^T
    p.idesc_bf16 = bf16;                                 // dP = dO V^T
    p.idesc_bf16_mn = bf16 | (1u << 16);                 // dV += P^T dO
    p.idesc_ds_mn = (qk_f16 ? f16 : bf16) | (1u << 16);  // dQ += dS K, dK += dS^T Q (dS in the q/k type)
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
