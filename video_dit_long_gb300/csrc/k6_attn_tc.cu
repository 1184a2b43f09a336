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
// How (one CTA per work unit = 256 query rows of one (batch, head, chunk)):
//   warp 8      TMA producer (warps 8-11 form the control warpgroup, which
//               gives registers to the two softmax warpgroups): Q0/Q1 (2 x 128 rows) once, then K_j, V_j tiles of
//               128 keys x 128 dims through a 4-slot ring (32 KB per tile, two
//               128-byte-swizzled 64-dim panels per tile).
//   warps 9, 10 MMA issuers, one thread each, for Q tile 0 and Q tile 1:
//               S_i = Q_i K_j^T (SS, K-major) into TMEM, then O_i += P_i V_j
//               with P_i read from TMEM (TS) and V MN-major from shared
//               memory.  Each thread issues its tile's chain in order,
//               P_i.V(j) then S_i(j+1); the tensor pipe interleaves the two
//               chains, so each softmax group has the other tile's MMAs to
//               hide behind.
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

#include "k6_attn_common.cuh"
#include "k6_device.cuh"
#include "k6_internal.h"

namespace k6 {

namespace tc {
constexpr int NSTAGE = 4;                     // K/V tile slots
constexpr int SMEM_Q = 0;
constexpr int SMEM_KV = NQ * TILE;
constexpr int SMEM_BAR = SMEM_KV + NSTAGE * TILE;
constexpr int P_PARTS = 2;                    // P of a tile is published in this many parts
constexpr int KP = BN / P_PARTS;              // keys per part
constexpr int MMA_PER_PART = KP / 16;         // P.V MMAs (K = 16 keys each) per part
constexpr int NBAR = 1 + 2 * NSTAGE + NQ + NQ * P_PARTS + NQ + NQ + 1;  // q_full, kv_full/empty, s_full,
                                                                       // p parts, o_final, o_step, drain
constexpr int SMEM_TOTAL = SMEM_BAR + NBAR * 8 + 16;
constexpr int SMEM_ALLOC = SMEM_TOTAL + 1024;  // room to align the base to 1024 bytes
constexpr int THREADS = 384;                  // 3 warpgroups: softmax 0, softmax 1, producer/MMA/spare
// Register split (launch: 384 x 168 = 64512): softmax groups grow to 184,
// the producer/MMA group shrinks to 136: 2*128*184 + 128*136 = 64512.
constexpr int REGS_SOFTMAX = 184;
constexpr int REGS_CONTROL = 136;
constexpr int TMEM_COLS = 512;
}  // namespace tc

// Each CTA loads its Q tile pair once and runs its chunks one after another;
// the K/V ring, the barrier phases and tensor memory carry over from one chunk
// to the next, so the next chunk's first Q.K^T overlaps the previous chunk's
// last P.V and epilogue.
// MERGE (p.merge): the CTA's consecutive chunks leave one partial instead of
// one each.  Their log-sum-exp merge is done in tensor memory as it goes: the
// row max, row sum and unnormalised O of the chunks so far carry into the next
// chunk, whose tiles rescale them exactly as later tiles of one chunk do
// (combining (m_a, l_a, O_a) with (m_b, l_b, O_b) under m = max(m_a, m_b) is
// the merge out = sum_c exp(LSE_c - LSE) O_c with LSE = m + ln l).  Only the
// group's last chunk runs the epilogue.
// BOUNDED: constant-max softmax.  Each row's running max is replaced by the
// precomputed bound p.row_bound (>= every logit of the row), so the softmax
// takes no row maximum and never rescales O; a row whose every term
// underflows (a bound far above the true maximum) is reported as DEV_RANGE.
// QK8: q/k/joint_k are e4m3.  Their tiles are 128 rows of 128 bytes (one
// swizzle panel, 16 KB, in the first half of their 32 KB slots) and Q.K^T runs
// as 4 kind::f8f6f4 MMAs of K = 32 per tile instead of 8 kind::f16 MMAs; P.V is
// unchanged (bf16 P from tensor memory, bf16 V).
template <bool BOUNDED, bool QK8>
__global__ void __launch_bounds__(tc::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_jk,
                   const __grid_constant__ CUtensorMap tm_jv, const TcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SMEM_BAR);
    uint64_t *q_full = bars;
    uint64_t *kv_full = q_full + 1;
    uint64_t *kv_empty = kv_full + NSTAGE;
    uint64_t *s_full = kv_empty + NSTAGE;
    uint64_t *p_part = s_full + NQ;  // [NQ][P_PARTS]
    uint64_t *o_final = p_part + NQ * P_PARTS;
    uint64_t *o_step = o_final + NQ;
    uint64_t *drain = o_step + NQ;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NSTAGE; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], NQ);  // released by both Q tiles' issuers
        }
        for (int i = 0; i < NQ; i++) {
            mbar_init(&s_full[i], 1);
            for (int q = 0; q < P_PARTS; q++) mbar_init(&p_part[i * P_PARTS + q], BM);
            mbar_init(&o_final[i], 1);
            mbar_init(&o_step[i], 1);
        }
        mbar_init(drain, NQ);  // one commit per MMA issuer
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
        if (warp == 8 && lane == 0) {
            // -------------------------------------------------- TMA producer
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_jk);
            prefetch_tmap(&tm_jv);
            uint32_t kv_idx = 0;  // K/V tile loads issued so far (K_j, V_j alternate)
            uint32_t uc = 0;      // units started by this CTA
            bool ok = true;
            const long u0 = (long)blockIdx.x * p.group, u1 = u0 + p.group;
            for (long u = u0; u < u1 && ok; u++, uc++) {
                const Unit un = decode_unit(p, u);
                const TileRange tr = chunk_tiles(p, un.c);
                if (uc == 0) {  // the CTA's Q tile pair, once
                    mbar_arrive_expect_tx(q_full, NQ * (QK8 ? PANEL : TILE));
                    for (int i = 0; i < NQ; i++)
                        for (int half = 0; half < (QK8 ? 1 : 2); half++)
                            tma_load_4d(smem + SMEM_Q + i * TILE + half * PANEL, &tm_q, q_full, half * 64, un.h,
                                        un.q0 + i * BM, un.b);
                }
                for (int j = 0; j < tr.T && ok; j++) {
                    int map, row, valid;
                    tr.at(j, map, row, valid);
                    for (int kv = 0; kv < 2; kv++, kv_idx++) {
                        const uint32_t slot = kv_idx % NSTAGE;
                        if (!mbar_wait(&kv_empty[slot], ((kv_idx / NSTAGE) & 1) ^ 1, w)) {
                            ok = false;
                            break;
                        }
                        const CUtensorMap *tm = kv == 0 ? (map == 0 ? &tm_k : &tm_jk) : (map == 0 ? &tm_v : &tm_jv);
                        const bool one_panel = QK8 && kv == 0;  // an e4m3 K tile is one 16 KB panel
                        mbar_arrive_expect_tx(&kv_full[slot], one_panel ? PANEL : TILE);
                        uint8_t *dst = smem + SMEM_KV + slot * TILE;
                        tma_load_4d(dst, tm, &kv_full[slot], 0, un.h, row, un.b);
                        if (!one_panel) tma_load_4d(dst + PANEL, tm, &kv_full[slot], 64, un.h, row, un.b);
                    }
                }
            }
            // let every copy issued into shared memory land before the CTA can exit
            if (uc > 0) mbar_drain(q_full, 0, DRAIN_NS);
            for (uint32_t idx = kv_idx > NSTAGE ? kv_idx - NSTAGE : 0; idx < kv_idx; idx++)
                mbar_drain(&kv_full[idx % NSTAGE], (idx / NSTAGE) & 1, DRAIN_NS);
        } else if ((warp == 9 || warp == 10) && lane == 0) {
            // -------------------------------------------------- MMA issuers
            // One issuing thread per Q tile, on two different SM sub-partitions.
            // Each sub-partition also runs two softmax warps, whose issue slots
            // a single issuing thread would share: it then issues an MMA about
            // every 90 cycles against the 64 the tensor pipe takes for one, and
            // the pipe starves.  Two issuers keep it fed.  Tile i's S_i and P_i.V
            // form one accumulator chain issued by one thread in order, so the
            // two threads never have to be ordered against each other; a K or V
            // slot is read by both tiles and is released by both (kv_empty
            // counts two arrivals).
            const int i = warp - 9;  // the Q tile this thread issues for
            const uint32_t idesc_qk = p.idesc_qk;
            const uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
            const uint32_t sQ = smem_u32(smem + SMEM_Q);
            // Descriptors are built once; per MMA only the start-address field
            // (bits 0-13, 16-byte units) moves, so each issue is one 64-bit add.
            const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);                       // Q / K: K-major, SBO 1024
            const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + SMEM_KV), PANEL, 1024);  // V: MN-major, LBO = panel
            const uint64_t qa = dq0 + ((uint64_t)(i * TILE) >> 4);
            const uint32_t tS = tmem + i * BN, tO = tmem + 2 * BN + i * D;
            // S_i = Q_i K^T from the K tile in `slot`: steps of 16 (bf16/fp16) or 32 (e4m3) head dims
            auto issue_s = [&](uint32_t slot) {
                const uint64_t kb = dq0 + ((uint64_t)(SMEM_KV - SMEM_Q + slot * TILE) >> 4);
                if constexpr (QK8) {
#pragma unroll
                    for (int kk = 0; kk < D / 32; kk++) {
                        const uint64_t off = (uint64_t)(kk * 32) >> 4;
                        mma_ss_f8(tS, qa + off, kb + off, idesc_qk, kk > 0);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++) {
                        const uint64_t off = (uint64_t)((kk >> 2) * PANEL + (kk & 3) * 32) >> 4;
                        mma_ss(tS, qa + off, kb + off, idesc_qk, kk > 0);
                    }
                }
            };
            // keys [16*k0, 16*k1) of O_i += P_i . V from the V tile in `slot`
            auto issue_pv = [&](uint32_t slot, bool acc, int k0, int k1) {
                const uint64_t vb = dv0 + ((uint64_t)(slot * TILE) >> 4);
#pragma unroll
                for (int kk = k0; kk < k1; kk++)
                    mma_ts(tO, tS + kk * 8, vb + ((uint64_t)(kk * 16 * 128) >> 4), idesc_pv,
                           (acc || kk > 0) ? 1u : 0u);
            };
            uint32_t step_phase = 0;
            // P_i lives in S_i's columns: in strict mode let the P.V that read it finish before S_i is rewritten
            auto strict_wait = [&]() -> bool {
                if (!p.strict_order) return true;
                tc_commit(&o_step[i]);
                const bool done = mbar_wait(&o_step[i], step_phase, w);
                step_phase ^= 1;
                return done;
            };
            uint32_t kv_idx = 0;  // K/V tiles consumed (K_j, V_j alternate)
            uint32_t tile = 0;    // K/V tiles finished over all units: phase of s_full / p_part
            uint32_t uc = 0;
            bool started = false;  // any P.V issued yet (the strict hazard exists from then on)
            bool ok = true;
            const long u0 = (long)blockIdx.x * p.group, u1 = u0 + p.group;
            for (long u = u0; u < u1 && ok; u++, uc++) {
                const Unit un = decode_unit(p, u);
                const int T = chunk_tiles(p, un.c).T;
                const bool carry = p.merge && uc > 0;      // O accumulates over the previous chunks
                const bool last = !p.merge || u + 1 == u1;  // this chunk's O goes to the epilogue
                ok = (uc > 0 || mbar_wait(q_full, 0, w)) &&
                     mbar_wait(&kv_full[kv_idx % NSTAGE], (kv_idx / NSTAGE) & 1, w);
                if (!ok) break;
                tc_fence_after();
                if (started && !(ok = strict_wait())) break;
                issue_s(kv_idx % NSTAGE);
                tc_commit(&s_full[i]);
                tc_commit(&kv_empty[kv_idx % NSTAGE]);
                // Per K/V tile j: P_i.V(j), part by part as the softmax publishes
                // P_i, then S_i(j+1), which overwrites P_i(j) and so follows it.
                for (int j = 0; j < T && ok; j++) {
                    const uint32_t vidx = kv_idx + 2 * j + 1, kidx = vidx + 1;
                    const uint32_t vs = vidx % NSTAGE, ks = kidx % NSTAGE;
                    const uint32_t ph = (tile + j) & 1;
                    if (!(ok = mbar_wait(&kv_full[vs], (vidx / NSTAGE) & 1, w))) break;
                    for (int q = 0; q < P_PARTS && ok; q++) {
                        if (!(ok = mbar_wait(&p_part[i * P_PARTS + q], ph, w))) break;
                        tc_fence_after();
                        issue_pv(vs, carry || j > 0 || q > 0, q * MMA_PER_PART, (q + 1) * MMA_PER_PART);
                    }
                    if (!ok) break;
                    started = true;
                    if (last && j + 1 == T) tc_commit(&o_final[i]);
                    tc_commit(&kv_empty[vs]);
                    if (j + 1 == T) continue;
                    if (!(ok = strict_wait())) break;
                    if (!(ok = mbar_wait(&kv_full[ks], (kidx / NSTAGE) & 1, w))) break;
                    tc_fence_after();
                    issue_s(ks);
                    tc_commit(&s_full[i]);
                    tc_commit(&kv_empty[ks]);
                }
                kv_idx += 2 * T;
                tile += T;
            }
            // every MMA issued so far must complete before tensor memory is freed
            // (the drain barrier counts one arrival per issuer)
            tc_commit(drain);
            mbar_drain(drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        regs_increase<REGS_SOFTMAX>();
        // ------------------------------------------------ softmax / epilogue
        const int i = warp / 4;                       // Q tile of this warpgroup
        const int r = threadIdx.x % BM;               // row within the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
        const uint32_t tS = lane_base + i * BN;
        const uint32_t tO = lane_base + 2 * BN + i * D;
        const float sl2 = p.scale_log2;
        uint32_t tile = 0, uc = 0, n_epi = 0;
        bool ok = true;
        float m_run = -INFINITY, l_run = 0.f;
        const long u0 = (long)blockIdx.x * p.group, u1 = u0 + p.group;
        for (long u = u0; u < u1 && ok; u++, uc++) {
            const Unit un = decode_unit(p, u);
            const TileRange tr = chunk_tiles(p, un.c);
            const int T = tr.T;
            const bool carry = p.merge && uc > 0;      // (m, l, O) of the previous chunks carry over
            const bool last = !p.merge || u + 1 == u1;
            if (!carry) m_run = -INFINITY, l_run = 0.f;
            const long grow_u = (long)un.q0 + i * BM + r;
            if constexpr (BOUNDED)
                m_run = grow_u < p.Sq ? p.row_bound[((long)un.b * p.H + un.h) * p.Sq + grow_u] * 1.4426950408889634f
                                      : 0.f;
            for (int j = 0; j < T; j++) {
                int map, row, valid;
                tr.at(j, map, row, valid);
                if (!mbar_wait(&s_full[i], (tile + j) & 1, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[BN];
#pragma unroll
                for (int cc = 0; cc < BN / 32; cc++)
                    tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
                tmem_ld_wait();
                bool rescale = false;  // warp-uniform
                float alpha = 1.f;
                if (valid < BN) {  // ragged tile end (warp-uniform): keys past the segment get -inf
#pragma unroll
                    for (int k = 0; k < BN; k++)
                        if (k >= valid) s[k] = 0xff800000u;
                }
                if constexpr (!BOUNDED) {
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
                if (j == 0 && !carry) m_run = mt;
                else need = mt > m_run + RESCALE_THRESHOLD;
                if (__any_sync(0xffffffffu, need)) {
                    // O_i holds P.V of tiles < j (S_i(j) was committed after it); it is
                    // rescaled below, after the first part of P is stored, before P.V(j)
                    rescale = true;
                    if (need) {
                        alpha = ex2(m_run - mt);
                        m_run = mt;
                        l_run *= alpha;
                    }
                }
                }
                // p = 2^(s * scale*log2e - m): packed FMA, then the SFU; row sum on
                // packed adds.  P is published in parts so that P.V can start on
                // the first keys while the rest is computed.
                const uint64_t scale2 = f2(sl2, sl2), negm2 = f2(-m_run, -m_run);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int q = 0; q < P_PARTS; q++) {
                    uint32_t pk[KP / 2];
#pragma unroll
                    for (int k = 0; k < KP; k += 2) {
                        const int kk = q * KP + k;
                        float a, b2;
                        f2_split(ffma2(f2(__uint_as_float(s[kk]), __uint_as_float(s[kk + 1])), scale2, negm2), a,
                                 b2);
                        const float p0 = ex2(a), p1 = ex2(b2);
                        pk[k / 2] = pack_bf16x2(p0, p1);
                        acc[(k / 2) & 3] = fadd2(acc[(k / 2) & 3], f2(p0, p1));
                    }
                    tmem_st_cols<KP / 2>(tS + q * (KP / 2), pk);
                    if (!BOUNDED && q == 0 && rescale) {
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
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&p_part[i * P_PARTS + q]);
                }
                float sum;
                {
                    float a0, a1, b0, b1;
                    f2_split(fadd2(acc[0], acc[1]), a0, a1);
                    f2_split(fadd2(acc[2], acc[3]), b0, b1);
                    sum = (a0 + a1) + (b0 + b1);
                }
                l_run += sum;
            }
            if (!last) {  // the group's partial is written after its last chunk
                tile += T;
                continue;
            }
            if (!ok || !mbar_wait(&o_final[i], n_epi & 1, w)) {
                ok = false;
                break;
            }
            n_epi++;
            const long pc = p.merge ? un.c / p.group : un.c;  // index of the partial written
            // epilogue: O_i / l to the output (or fp32 partial), LSE; the next
            // unit's first P.V into O_i waits for this warpgroup's next P
            tc_fence_after();
            const long grow = (long)un.q0 + i * BM + r;
            const bool live = grow < p.Sq;
            if constexpr (BOUNDED) {
                if (live && !(l_run > 0.f)) atomicCAS(p.err, DEV_OK, DEV_RANGE);  // bound too loose: all terms underflowed
            }
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const long obase = (((long)un.b * p.Sq + (live ? grow : 0)) * p.H + un.h) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; cc++) {
                uint32_t o[32];
                tmem_ld32(tO + cc * 32, o);
                tmem_ld_wait();
                if (live) {
                    if (p.out_f32) {
                        float *dst = static_cast<float *>(p.out) + (long long)pc * p.o_stride + obase + cc * 32;
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
                            // streaming stores: the partials are read once, by the merge, and should
                            // not push this chunk's K/V out of L2
                            __stcs(reinterpret_cast<float4 *>(dst + k),
                                   make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                                               __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv));
                    } else {
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + obase + cc * 32;
#pragma unroll
                        for (int k = 0; k < 32; k += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv);
                            v.y = pack_bf16x2(__uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
                            v.z = pack_bf16x2(__uint_as_float(o[k + 4]) * inv, __uint_as_float(o[k + 5]) * inv);
                            v.w = pack_bf16x2(__uint_as_float(o[k + 6]) * inv, __uint_as_float(o[k + 7]) * inv);
                            *reinterpret_cast<uint4 *>(dst + k) = v;
                        }
                    }
                }
            }
            if (live && p.lse)
                p.lse[(long long)pc * p.l_stride + ((long)un.b * p.H + un.h) * p.Sq + grow] =
                    (m_run + log2f(l_run)) * 0.69314718055994531f;
            tile += T;
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

cudaError_t launch_attn_tc(const Geom &g, const void *q, const void *k, const void *v, const void *jk,
                           const void *jv, int n_chunks, void *out, float *lse, const AttnTcOptions &opt,
                           cudaStream_t st, const char **why) {
    CUtensorMap mq, mk, mv, mjk, mjv;
    const bool has_joint = g.Nj > 0;
    const bool has_video = g.Nv > 0;
    // an empty segment never issues loads; give its maps a valid stand-in
    const void *kk = has_video ? k : jk, *vv = has_video ? v : jv;
    const long kv_rows = has_video ? g.Nv : g.Nj;
    // the tile copies move 2-byte elements (fp16 q/k travel through the same maps), or 1-byte e4m3 q/k
    const int qkb = opt.qk8 ? 1 : 2;
    if (!make_bshd_map(&mq, q, g.Sq, g.H, g.B, false, why, qkb) ||
        !make_bshd_map(&mk, kk, kv_rows, g.H, g.B, false, why, has_video ? qkb : 2) ||
        !make_bshd_map(&mv, vv, kv_rows, g.H, g.B, false, why) ||
        !make_bshd_map(&mjk, has_joint ? jk : kk, has_joint ? g.Nj : kv_rows, g.H, g.B, false, why,
                       has_joint || has_video ? qkb : 2) ||
        !make_bshd_map(&mjv, has_joint ? jv : vv, has_joint ? g.Nj : kv_rows, g.H, g.B, false, why))
        return cudaErrorInvalidValue;
    auto kernel = opt.qk8 ? (opt.row_bound ? attn_tc_kernel<true, true> : attn_tc_kernel<false, true>)
                          : (opt.row_bound ? attn_tc_kernel<true, false> : attn_tc_kernel<false, false>);
    cudaError_t attr_err = set_max_dynamic_smem((const void *)kernel, tc::SMEM_ALLOC);
    if (attr_err != cudaSuccess) return attr_err;
    TcParams p;
    p.S = g.S;
    p.Sq = g.Sq;
    p.Nv = g.Nv;
    p.Nj = g.Nj;
    p.H = g.H;
    p.n_chunks = n_chunks;
    p.unit_rows = tc::NQ * tc::BM;
    p.q_pairs = (int)((g.Sq + p.unit_rows - 1) / p.unit_rows);
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.d));
    p.out = out;
    p.lse = lse;
    p.o_stride = (long long)g.B * g.Sq * g.H * g.d;
    p.l_stride = (long long)g.B * g.H * g.Sq;
    p.wait_limit_ns = opt.wait_limit_ns;
    p.err = opt.err;
    p.strict_order = opt.strict_order;
    // Q.K^T operands: bf16 (A/B format 1), fp16 (format 0) or e4m3 (kind::f8f6f4, format 0); P.V stays bf16
    p.idesc_qk = opt.qk8      ? idesc_e4m3_f32(tc::BM, tc::BN)
                 : opt.qk_f16 ? (idesc_bf16_f32(tc::BM, tc::BN, false) & ~((7u << 7) | (7u << 10)))
                              : idesc_bf16_f32(tc::BM, tc::BN, false);
    p.units = (long)g.B * g.H * n_chunks * p.q_pairs;
    if (p.units == 0) return cudaSuccess;
    if (p.units >= (1L << 31)) {
        if (why) *why = "too many work units (batch x heads x chunks x query-tile pairs must stay below 2^31)";
        return cudaErrorInvalidValue;
    }
    // chunks per CTA (sharing one load of Q): the caller's group, else the
    // library's choice (chunk_group); with merge the group leaves one partial
    p.group = opt.group > 0 ? opt.group : chunk_group(g, n_chunks);
    if (n_chunks % p.group) {
        if (why) *why = "the chunk group must divide the chunk count";
        return cudaErrorInvalidValue;
    }
    p.merge = opt.merge && p.group > 1;
    p.out_f32 = (p.merge ? n_chunks / p.group : n_chunks) > 1;
    // One CTA per Q tile pair and chunk group: the block scheduler hands each
    // freed SM the next CTA, which keeps the CTAs in flight (and their K/V in
    // L2) in a tight window; measured faster than a static persistent
    // round-robin over SMs.
    const long grid = p.units / p.group;
    p.row_bound = opt.row_bound;
    kernel<<<(unsigned)grid, tc::THREADS, tc::SMEM_ALLOC, st>>>(mq, mk, mv, mjk, mjv, p);
    return cudaGetLastError();
}

}  // namespace k6
