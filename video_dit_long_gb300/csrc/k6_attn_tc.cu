// k6_attn_tc.cu -- bf16 joint-sequence attention on the 5th-generation tensor
// cores of sm_103a (tcgen05 MMA into tensor memory, TMA tile loads).
//
// What it computes: for one K/V chunk c of the joint sequence (video keys
// followed by the text/audio "joint tensors", xDiT PR #586 "How?"), every
// query row i gets
//   O_c[i] = sum_j softmax_j(q_i . k_j / sqrt(d)) v_j,  LSE_c[i] = log sum_j exp(q_i . k_j / sqrt(d)),
// full and non-causal ("Context Parallelism in vLLM Omni Neuron",
// "Self-Attention with Context Parallelism": local Q x full K/V; "Ring
// attention (current implementation)": one K/V chunk per ring step, partials
// combined through their log-sum-exp).  With one chunk the normalised output
// is written as bf16; with several, fp32 partials and LSE go to the caller's
// workspace for the merge kernel.
//
// How (one CTA = one work unit = 256 query rows of one (batch, head, chunk)):
//   warp 8      TMA producer (warps 8-11 form the control warpgroup, which
//               gives registers to the two softmax warpgroups): Q0/Q1 (2 x 128 rows) once, then K_j, V_j tiles of
//               128 keys x 128 dims through a 4-slot ring (32 KB per tile, two
//               128-byte-swizzled 64-dim panels per tile).
//   warp 9      MMA issuer (one thread): S_i = Q_i K_j^T (SS, K-major) into
//               TMEM, then O_i += P_i V_j with P_i read from TMEM (TS) and V
//               MN-major from shared memory.  Order per K/V tile:
//               PV0(j), S0(j+1), PV1(j), S1(j+1), so each softmax group has a
//               full P.V + S of the other group to hide behind.
//   warps 0-3   softmax of Q tile 0, warps 4-7 of Q tile 1: one thread per
//               query row (its TMEM lane); online softmax in base 2 with the
//               scale folded in; the running max is only moved (and O
//               rescaled in TMEM) when it grows by more than 2^8; P is packed
//               to bf16 and stored over the first 64 columns of its S tile.
//   Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.
//   The K/V range of a chunk is split into its video segment and its joint
//   segment (separate tensor maps); ragged tile ends are masked to -inf.
//   All mbarrier waits are bounded (globaltimer); a wait that runs out sets
//   the handle's error word and every warp leaves in order, letting copies
//   and MMAs in flight land before tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "k6_device.cuh"
#include "k6_internal.h"

namespace k6 {

namespace tc {
constexpr int D = 128;
constexpr int BM = 128;                       // query rows per Q tile
constexpr int BN = 128;                       // keys per K/V tile
constexpr int NQ = 2;                         // Q tiles per CTA
constexpr int NSTAGE = 4;                     // K/V tile slots
constexpr int PANEL = BM * 64 * 2;            // one 128-row x 64-dim bf16 panel: 16 KB
constexpr int TILE = 2 * PANEL;               // 32 KB
constexpr int SMEM_Q = 0;
constexpr int SMEM_KV = NQ * TILE;
constexpr int SMEM_BAR = SMEM_KV + NSTAGE * TILE;
constexpr int NBAR = 1 + 2 * NSTAGE + 3 * NQ + NQ + 1;  // q_full, kv_full/empty, s/p/o_final, o_step, drain
constexpr int SMEM_TOTAL = SMEM_BAR + NBAR * 8 + 16;
constexpr int SMEM_ALLOC = SMEM_TOTAL + 1024;  // room to align the base to 1024 bytes
constexpr int THREADS = 384;                  // 3 warpgroups: softmax 0, softmax 1, producer/MMA/spare
// Register split (launch: 384 x 168 = 64512): softmax groups grow to 200,
// the producer/MMA group shrinks to 104: 2*128*200 + 128*104 = 64512.
constexpr int REGS_SOFTMAX = 200;
constexpr int REGS_CONTROL = 104;
constexpr int TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.0f;     // log2 units: rescale when the max grows past 2^8
constexpr unsigned long long DRAIN_NS = 1000000000ull;
}  // namespace tc

struct TcParams {
    long S, Nv, Nj;
    int H, n_chunks, q_pairs;
    float scale_log2;                         // log2(e) / sqrt(d)
    void *out;                                // bf16 [B][S][H][d] or fp32 partials
    float *lse;
    int out_f32;
    long long o_stride, l_stride;             // elements between chunks
    unsigned long long wait_limit_ns;
    int *err;
    int strict_order;
    uint32_t idesc_qk;                        // instruction descriptor of Q.K^T (bf16 or fp16 operands)
};

// K/V tile j of a chunk: which tensor map (0 video, 1 joint), first row, valid keys.
struct TileRange {
    long v_beg, v_end, j_beg, j_end;
    int Tv, T;
    __device__ void at(int j, int &map, int &row, int &valid) const {
        if (j < Tv) {
            map = 0;
            long r = v_beg + (long)j * tc::BN;
            row = (int)r;
            valid = (int)min((long)tc::BN, v_end - r);
        } else {
            map = 1;
            long r = j_beg + (long)(j - Tv) * tc::BN;
            row = (int)r;
            valid = (int)min((long)tc::BN, j_end - r);
        }
    }
};

__device__ __forceinline__ TileRange chunk_tiles(const TcParams &p, int c) {
    TileRange t;
    const long L = (p.S) / p.n_chunks;
    const long kb = (long)c * L, ke = kb + L;
    t.v_beg = kb;
    t.v_end = ke < p.Nv ? ke : p.Nv;
    t.j_beg = (kb > p.Nv ? kb : p.Nv) - p.Nv;
    t.j_end = ke > p.Nv ? ke - p.Nv : 0;
    t.Tv = t.v_end > t.v_beg ? (int)((t.v_end - t.v_beg + tc::BN - 1) / tc::BN) : 0;
    const int Tj = t.j_end > t.j_beg ? (int)((t.j_end - t.j_beg + tc::BN - 1) / tc::BN) : 0;
    t.T = t.Tv + Tj;
    return t;
}

__global__ void __launch_bounds__(tc::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_jk,
                   const __grid_constant__ CUtensorMap tm_jv, const TcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SMEM_BAR);
    uint64_t *q_full = bars;
    uint64_t *kv_full = bars + 1;
    uint64_t *kv_empty = kv_full + NSTAGE;
    uint64_t *s_full = kv_empty + NSTAGE;
    uint64_t *p_full = s_full + NQ;
    uint64_t *o_final = p_full + NQ;
    uint64_t *o_step = o_final + NQ;
    uint64_t *drain = o_step + NQ;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // work unit: (b, h, chunk, query-tile pair), pairs fastest so that CTAs
    // running together share one chunk's K/V in L2
    long unit = blockIdx.x;
    const int qp = (int)(unit % p.q_pairs);
    unit /= p.q_pairs;
    const int c = (int)(unit % p.n_chunks);
    unit /= p.n_chunks;
    const int h = (int)(unit % p.H);
    const int b = (int)(unit / p.H);
    const int q0 = qp * (NQ * BM);
    const TileRange tr = chunk_tiles(p, c);
    const int T = tr.T;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NSTAGE; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < NQ; i++) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], BM);
            mbar_init(&o_final[i], 1);
            mbar_init(&o_step[i], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{p.wait_limit_ns, p.err, abort_flag};

    if (warp >= 8) {
        regs_decrease<REGS_CONTROL>();
        if (warp == 8) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_jk);
            prefetch_tmap(&tm_jv);
            mbar_arrive_expect_tx(q_full, NQ * TILE);
            for (int i = 0; i < NQ; i++)
                for (int half = 0; half < 2; half++)
                    tma_load_4d(smem + SMEM_Q + i * TILE + half * PANEL, &tm_q, q_full, half * 64, h, q0 + i * BM, b);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < T && ok; j++) {
                int map, row, valid;
                tr.at(j, map, row, valid);
                for (int kv = 0; kv < 2; kv++) {
                    const int idx = 2 * j + kv, slot = idx % NSTAGE;
                    if (!mbar_wait(&kv_empty[slot], ((idx / NSTAGE) & 1) ^ 1, w)) {
                        ok = false;
                        break;
                    }
                    const CUtensorMap *tm = kv == 0 ? (map == 0 ? &tm_k : &tm_jk) : (map == 0 ? &tm_v : &tm_jv);
                    mbar_arrive_expect_tx(&kv_full[slot], TILE);
                    uint8_t *dst = smem + SMEM_KV + slot * TILE;
                    tma_load_4d(dst, tm, &kv_full[slot], 0, h, row, b);
                    tma_load_4d(dst + PANEL, tm, &kv_full[slot], 64, h, row, b);
                    issued++;
                }
            }
            // let every copy issued into shared memory land before the CTA can exit
            mbar_drain(q_full, 0, DRAIN_NS);
            for (int idx = issued > NSTAGE ? issued - NSTAGE : 0; idx < issued; idx++)
                mbar_drain(&kv_full[idx % NSTAGE], (idx / NSTAGE) & 1, DRAIN_NS);
        }
        __syncwarp();
        } else if (warp == 9) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = p.idesc_qk;
            const uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
            const uint32_t sQ = smem_u32(smem + SMEM_Q), sKV = smem_u32(smem + SMEM_KV);
            auto issue_s = [&](int i, int slot) {
                const uint32_t qa = sQ + i * TILE, kb = sKV + slot * TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;
                    mma_ss(tmem + i * BN, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
                           idesc_qk, kk > 0);
                }
            };
            auto issue_pv = [&](int i, int slot, bool acc) {
                const uint32_t vb = sKV + slot * TILE;
#pragma unroll
                for (int kk = 0; kk < BN / 16; kk++) {
                    mma_ts(tmem + 2 * BN + i * D, tmem + i * BN + kk * 8,
                           smem_desc_sw128(vb + kk * 16 * 128, PANEL, 1024), idesc_pv, (acc || kk > 0) ? 1u : 0u);
                }
            };
            uint32_t step_phase0 = 0, step_phase1 = 0;
            bool ok = mbar_wait(q_full, 0, w) && mbar_wait(&kv_full[0], 0, w);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                tc_commit(&s_full[0]);
                issue_s(1, 0);
                tc_commit(&s_full[1]);
                tc_commit(&kv_empty[0]);
            }
            // P.V of Q tile i for K/V tile j, then (if another tile follows) S_i(j+1)
            auto pv_then_s = [&](int i, int j, int vs, int ks, int kidx, uint32_t &step_phase) -> bool {
                if (!mbar_wait(&p_full[i], j & 1, w)) return false;
                tc_fence_after();
                issue_pv(i, vs, j > 0);
                if (i == NQ - 1) tc_commit(&kv_empty[vs]);
                if (j + 1 >= T) {
                    tc_commit(&o_final[i]);
                    return true;
                }
                if (p.strict_order) {
                    // P_i lives in S_i's columns: let P.V finish reading it first
                    tc_commit(&o_step[i]);
                    const bool done = mbar_wait(&o_step[i], step_phase, w);
                    step_phase ^= 1;
                    if (!done) return false;
                }
                if (i == 0) {
                    if (!mbar_wait(&kv_full[ks], (kidx / NSTAGE) & 1, w)) return false;
                    tc_fence_after();
                }
                issue_s(i, ks);
                tc_commit(&s_full[i]);
                if (i == NQ - 1) tc_commit(&kv_empty[ks]);
                return true;
            };
            for (int j = 0; j < T && ok; j++) {
                const int vidx = 2 * j + 1, vs = vidx % NSTAGE;
                const int kidx = 2 * j + 2, ks = kidx % NSTAGE;
                ok = mbar_wait(&kv_full[vs], (vidx / NSTAGE) & 1, w) && pv_then_s(0, j, vs, ks, kidx, step_phase0) &&
                     pv_then_s(1, j, vs, ks, kidx, step_phase1);
            }
            // every MMA issued so far must complete before tensor memory is freed
            tc_commit(drain);
            mbar_drain(drain, 0, DRAIN_NS);
        }
        __syncwarp();
        }
    } else {
        regs_increase<REGS_SOFTMAX>();
        // ------------------------------------------------ softmax / epilogue
        const int i = warp / 4;                       // Q tile of this warpgroup
        const int r = threadIdx.x % BM;               // row within the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
        const uint32_t tS = lane_base + i * BN;
        const uint32_t tO = lane_base + 2 * BN + i * D;
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; j++) {
            int map, row, valid;
            tr.at(j, map, row, valid);
            if (!mbar_wait(&s_full[i], j & 1, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[BN];
#pragma unroll
            for (int cc = 0; cc < BN / 32; cc++) tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
            tmem_ld_wait();
            if (valid < BN) {  // ragged tile end (warp-uniform): keys past the segment get -inf
#pragma unroll
                for (int k = 0; k < BN; k++)
                    if (k >= valid) s[k] = 0xff800000u;
            }
            // row max: four independent 3-input chains
            float mc[4];
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                const uint32_t *x = &s[c4 * 32];
                float m = fmax3(__uint_as_float(x[0]), __uint_as_float(x[1]), __uint_as_float(x[2]));
#pragma unroll
                for (int k = 3; k < 31; k += 2) m = fmax3(m, __uint_as_float(x[k]), __uint_as_float(x[k + 1]));
                mc[c4] = fmaxf(m, __uint_as_float(x[31]));
            }
            const float mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
            const float mt = mx * sl2;
            bool need = false;
            if (j == 0) m_run = mt;
            else need = mt > m_run + RESCALE_THRESHOLD;
            if (__any_sync(0xffffffffu, need)) {
                // O_i already holds P.V of tiles < j: S_i(j) was committed after it
                float alpha = 1.f;
                if (need) {
                    alpha = ex2(m_run - mt);
                    m_run = mt;
                    l_run *= alpha;
                }
#pragma unroll
                for (int cc = 0; cc < D / 32; cc++) {
                    uint32_t o[32];
                    tmem_ld32(tO + cc * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; k++) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st32(tO + cc * 32, o);
                }
            }
            // p = 2^(s * scale*log2e - m): packed FMA, then the SFU; row sum on packed adds
            const uint64_t scale2 = f2(sl2, sl2), negm2 = f2(-m_run, -m_run);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            uint32_t pk[BN / 2];
#pragma unroll
            for (int k = 0; k < BN; k += 2) {
                float a, b;
                f2_split(ffma2(f2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), scale2, negm2), a, b);
                const float p0 = ex2(a), p1 = ex2(b);
                pk[k / 2] = pack_bf16x2(p0, p1);
                acc[(k / 2) & 3] = fadd2(acc[(k / 2) & 3], f2(p0, p1));
            }
            float sum;
            {
                float a0, a1, b0, b1;
                f2_split(fadd2(acc[0], acc[1]), a0, a1);
                f2_split(fadd2(acc[2], acc[3]), b0, b1);
                sum = (a0 + a1) + (b0 + b1);
            }
            l_run += sum;
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[i]);
        }
        if (ok && T > 0 && mbar_wait(&o_final[i], 0, w)) {
            tc_fence_after();
            const long grow = (long)q0 + i * BM + r;
            const bool live = grow < p.S;
            const float inv = 1.f / l_run;
            const long obase = (((long)b * p.S + (live ? grow : 0)) * p.H + h) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; cc++) {
                uint32_t o[32];
                tmem_ld32(tO + cc * 32, o);
                tmem_ld_wait();
                if (live) {
                    if (p.out_f32) {
                        float *dst = static_cast<float *>(p.out) + (long long)c * p.o_stride + obase + cc * 32;
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
                            *reinterpret_cast<float4 *>(dst + k) =
                                make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                                            __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
                    } else {
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + obase + cc * 32;
#pragma unroll
                        for (int k = 0; k < 32; k += 8) {
                            uint4 u;
                            u.x = pack_bf16x2(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv);
                            u.y = pack_bf16x2(__uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
                            u.z = pack_bf16x2(__uint_as_float(o[k + 4]) * inv, __uint_as_float(o[k + 5]) * inv);
                            u.w = pack_bf16x2(__uint_as_float(o[k + 6]) * inv, __uint_as_float(o[k + 7]) * inv);
                            *reinterpret_cast<uint4 *>(dst + k) = u;
                        }
                    }
                }
            }
            if (live && p.lse)
                p.lse[(long long)c * p.l_stride + ((long)b * p.H + h) * p.S + grow] =
                    (m_run + log2f(l_run)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------- host

static PFN_cuTensorMapEncodeTiled_v12000 get_encode(const char **why) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn && why) *why = "cuTensorMapEncodeTiled is not available from the driver";
    return fn;
}

// Tensor map over a BSHD bf16 tensor [B][rows][H][128]: box = 64 dims x 1 head
// x 128 rows x 1 batch, 128-byte swizzle, zero fill out of bounds.
static bool make_map(CUtensorMap *m, const void *base, long rows, int H, int B, const char **why) {
    auto encode = get_encode(why);
    if (!encode) return false;
    cuuint64_t dims[4] = {(cuuint64_t)tc::D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)tc::D * 2, (cuuint64_t)H * tc::D * 2, (cuuint64_t)rows * H * tc::D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)tc::BM, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled rejected a tensor";
        return false;
    }
    return true;
}

cudaError_t launch_attn_tc(const Geom &g, const void *q, const void *k, const void *v, const void *jk,
                           const void *jv, int n_chunks, void *out, float *lse, const AttnTcOptions &opt,
                           cudaStream_t st, const char **why) {
    CUtensorMap mq, mk, mv, mjk, mjv;
    const bool has_joint = g.Nj > 0;
    const bool has_video = g.Nv > 0;
    // an empty segment never issues loads; give its maps a valid stand-in
    const void *kk = has_video ? k : jk, *vv = has_video ? v : jv;
    const long kv_rows = has_video ? g.Nv : g.Nj;
    if (!make_map(&mq, q, g.S, g.H, g.B, why) || !make_map(&mk, kk, kv_rows, g.H, g.B, why) ||
        !make_map(&mv, vv, kv_rows, g.H, g.B, why) ||
        !make_map(&mjk, has_joint ? jk : kk, has_joint ? g.Nj : kv_rows, g.H, g.B, why) ||
        !make_map(&mjv, has_joint ? jv : vv, has_joint ? g.Nj : kv_rows, g.H, g.B, why))
        return cudaErrorInvalidValue;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_ALLOC);
    });
    if (attr_err != cudaSuccess) return attr_err;
    TcParams p;
    p.S = g.S;
    p.Nv = g.Nv;
    p.Nj = g.Nj;
    p.H = g.H;
    p.n_chunks = n_chunks;
    p.q_pairs = (int)((g.S + tc::NQ * tc::BM - 1) / (tc::NQ * tc::BM));
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
    p.out = out;
    p.lse = lse;
    p.out_f32 = n_chunks > 1;
    p.o_stride = (long long)g.B * g.S * g.H * g.d;
    p.l_stride = (long long)g.B * g.H * g.S;
    p.wait_limit_ns = opt.wait_limit_ns;
    p.err = opt.err;
    p.strict_order = opt.strict_order;
    // Q.K^T operands: bf16 (A/B format 1) or fp16 (format 0); P.V stays bf16
    p.idesc_qk = opt.qk_f16 ? (idesc_bf16_f32(tc::BM, tc::BN, false) & ~((7u << 7) | (7u << 10)))
                            : idesc_bf16_f32(tc::BM, tc::BN, false);
    const long units = (long)g.B * g.H * n_chunks * p.q_pairs;
    if (units == 0) return cudaSuccess;
    attn_tc_kernel<<<(unsigned)units, tc::THREADS, tc::SMEM_ALLOC, st>>>(mq, mk, mv, mjk, mjv, p);
    return cudaGetLastError();
}

}  // namespace k6
