// k6_attn_single.cu -- joint-sequence attention on the 5th-generation tensor
// cores of sm_103a (tcgen05 MMA into tensor memory, TMA tile loads), one
// 128-row Q tile per CTA.
//
// What it computes: for one K/V chunk c of the joint sequence (video keys
// followed by the text/audio "joint tensors", xDiT PR #586 "How?"), every
// query row i gets
//   O_c[i] = sum_j softmax_j(q_i . k_j / sqrt(d)) v_j,  LSE_c[i] = log sum_j exp(q_i . k_j / sqrt(d)),
// full and non-causal ("Context Parallelism in vLLM Omni Neuron",
// "Self-Attention with Context Parallelism": local Q x full K/V; "Ring
// attention (current implementation)": one K/V chunk per ring step, partials
// combined through their log-sum-exp).  With one chunk (or one chunk group
// merged in the kernel) the normalised output is written as bf16; otherwise
// fp32 partials and LSE go to the caller's workspace for the merge kernel.
// q/k/joint_k are bf16, fp16 or e4m3 (QK8); v/joint_v bf16.
//
// How (one CTA per work unit = 128 query rows of one (batch, head), over a
// group of consecutive chunks):
//   warp 8      TMA producer: the Q tile once, then K_j and V_j tiles of 128
//               keys x 128 dims through a 6-slot ring of 32 KB slots (two
//               128-byte-swizzled 64-dim panels; an e4m3 tile is one panel),
//               in the order K_0 K_1 V_0 K_2 V_1 K_3 ..., so that K runs two
//               tiles ahead of V.
//   warp 9      issues every S(n) = Q K_n^T (SS, both K-major) into
//               tensor-memory buffer n % 3; the buffer held P(n-3), so S(n)
//               waits for the P.V of tile n-3 (pv_buf), and having seen it
//               done, frees V(n-3)'s ring slot (the softmax group that sees
//               S(n) done frees K(n)'s), so the issuers spend no commits on
//               the ring.
//   warp 10     issues every O += P(n) V_n (P from tensor memory, V MN-major
//               from shared memory), part by part as the softmax publishes
//               P(n).  Two issuers on different SM sub-partitions: one would
//               share its sub-partition's issue slots with two softmax warps
//               and feed the tensor pipe too slowly.
//   Warps 8-10 run whole and converged: every lane waits (a warp-uniform
//   vote), one lane picked by elect.sync issues each copy, MMA and commit.
//   With 16-bit q/k the CTAs run in clusters of two that share each K/V tile,
//   every CTA loading one panel for both (CLUSTER, below).
//   warps 0-7   two softmax warpgroups on alternate K/V tiles (whole rows, one
//               thread per row = TMEM lane), passing the running row max from
//               tile to tile; both run the epilogue, each writing half of O.
//   Tensor memory (512 columns): S buffers 0-2 (128 columns each), O.
//   With p.merge a CTA's group of chunks leaves one partial: (m, l, O) carry
//   from one chunk into the next and only the group's last chunk runs the
//   epilogue.
// All mbarrier waits are bounded (globaltimer); a wait that runs out records
// the error, sets the CTA's abort flag, and every warp leaves in order,
// letting copies and MMAs in flight land before tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>


#include "k6_attn_common.cuh"
#include "k6_device.cuh"
#include "k6_internal.h"

namespace k6 {

// 1: 16-bit q/k attention runs in CTA pairs that multicast K/V tiles.
#ifndef K6_KV_MULTICAST
#define K6_KV_MULTICAST 1
#endif

namespace ts {
using tc::BM;
using tc::BN;
using tc::D;
using tc::PANEL;
using tc::TILE;
// K/V tile slots.  Inside a unit the loads alternate K and V, so with an even
// count a slot keeps one kind there: K(n) reuses K(n-3)'s slot, freed once
// S(n-3) is done, and V(n) reuses V(n-3)'s, freed once P(n-3).V is done.
// (With five, K(n) took V(n-4)'s slot and could not load before P(n-4).V
// finished.)
constexpr int NSTAGE = 6;
// K_t is loaded before V_{t-KAHEAD} (see k_load, v_load).  Each slot's kv_full
// barrier is tested by phase parity only, so a consumer may wait for a load
// only once the slot's previous load has landed, or the wait could match that
// earlier phase.  In a unit's steady state the previous load of a slot is the
// same kind, waited for by the same warp before; at unit starts and tails the
// kinds shift, and a model of every warp's waits in program order checks that
// the rule still holds there, for every sequence of up to three chunks of 1-7
// tiles.  (With five slots the kinds alternate in a slot and a lead of 3
// breaks the rule.)
constexpr int KAHEAD = 2;
constexpr int NSBUF = 3;                      // S buffers in tensor memory
constexpr int SMEM_Q = 0;
constexpr int SMEM_KV = TILE;
constexpr int SMEM_BAR = SMEM_KV + NSTAGE * TILE;
constexpr int P_PARTS = 2;                    // P of a tile is published in this many parts
constexpr int KP = BN / P_PARTS;              // keys per part
// q_full, kv_full [source CTA][slot], kv_empty, s_full, p_part [S buffer][part], o_final, drain,
// pv_buf [S buffer], m_ready [tile parity][warp], epi [warp], epi_done [warp]
constexpr int NBAR = 1 + 3 * NSTAGE + NSBUF + NSBUF * P_PARTS + 1 + 1 + NSBUF + 8 + 4 + 4;
// + TMEM address word, abort flag and the count of K/V loads this CTA issued
constexpr int SMEM_XCH = (SMEM_BAR + NBAR * 8 + 16 + 15) & ~15;
// running row max [row]; epilogue exchange [warpgroup][row] of (l, m)
constexpr int SMEM_TOTAL = SMEM_XCH + (BM + 2 * 2 * BM) * 4;
// The tiles need a 1024-byte-aligned base (128-byte swizzle).  The dynamic
// shared memory of a kernel without static shared memory starts there; the
// kernel checks it and reports DEV_LAYOUT otherwise, as there is no room to
// realign: six 32 KB slots and the Q tile leave 96 of the 227 KB.
constexpr int SMEM_ALLOC = SMEM_TOTAL;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory plan exceeds the per-CTA limit");
constexpr int THREADS = 384;                  // softmax halves 0 and 1, producer/MMA/spare
// Register split (launch: 384 x 168 = 64512): 2*128*184 + 128*136 = 64512.
constexpr int REGS_SOFTMAX = 184;
constexpr int REGS_CONTROL = 136;
constexpr int TMEM_COLS = 512;
constexpr int O_COL = NSBUF * BN;             // O accumulator columns [384, 512)
}  // namespace ts

// Load order of a unit of T K/V tiles: K_0 .. K_{A-1}, then V_j followed by
// K_{j+A} (while j + A < T), A = KAHEAD: K runs A tiles ahead of V.  The
// index of each tile's load within the unit:
__device__ __forceinline__ uint32_t k_load(int t, int T) {
    (void)T;
    return t < ts::KAHEAD ? t : 2 * t - ts::KAHEAD + 1;
}
__device__ __forceinline__ uint32_t v_load(int j, int T) {
    const int lead = T < ts::KAHEAD ? T : ts::KAHEAD;      // K loads before V_0
    const int more = T > ts::KAHEAD ? T - ts::KAHEAD : 0;  // K loads that follow a V
    return lead + j + (j < more ? j : more);
}

// QK8: q/k/joint_k are e4m3.  Their tiles are 128 rows of 128 bytes (one
// swizzle panel, 16 KB, in the first half of their 32 KB slots) and Q.K^T runs as
// 4 kind::f8f6f4 MMAs of K = 32 per tile instead of 8 kind::f16 MMAs; P.V is
// unchanged (bf16 P from tensor memory, bf16 V).
//
// CLUSTER (16-bit q/k): the grid runs in clusters of two CTAs that hold
// consecutive Q tiles of the same (batch, head, chunk group), so they stream
// the same K/V tiles.  Each CTA loads one 64-dim panel of every tile (CTA rank
// r: panel r) and multicasts it to both, halving the K/V bytes read from L2.
// kv_full is split by source CTA; each CTA's producer arms both of its own
// barriers for a load when it issues its panel of it.  A slot is refilled only
// when the consumers of both CTAs have released it (kv_empty counts one local
// and one remote arrival).  On the way out, after a cluster barrier (no copy
// or remote arrival is issued any more), each CTA waits for the last load of
// every source in every slot to land, arming first a phase the partner sent
// but this CTA never armed, and a second cluster barrier keeps both CTAs
// resident until then.
template <bool BOUNDED, bool QK8, bool CLUSTER>
__global__ void __launch_bounds__(ts::THREADS, 1)
    attn_tc_single_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_jk,
                          const __grid_constant__ CUtensorMap tm_jv, const TcParams p) {
    using namespace ts;
    static_assert(!(CLUSTER && QK8), "the cluster form multicasts the two 64-dim panels of 16-bit tiles");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    if (smem_u32(smem) & 1023u) {  // the same for every thread: the CTA leaves before any barrier
        if (threadIdx.x == 0) atomicCAS(p.err, DEV_OK, DEV_LAYOUT);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SMEM_BAR);
    uint64_t *q_full = bars;
    uint64_t *kv_full = q_full + 1;        // [source CTA rank][slot]; rank 0 only without CLUSTER
    uint64_t *kv_empty = kv_full + 2 * NSTAGE;
    uint64_t *s_full = kv_empty + NSTAGE;  // [NSBUF]
    // [S buffer][part], 128 arrivals each.  Indexed by buffer, not by tile parity:
    // P(n+3), the next completion of the same barrier, needs S(n+3), which waits
    // for P(n).V, so the P.V thread can never miss a phase.  (By parity, P(n+2)
    // could complete the barrier a second time while that thread still waits for
    // a slow V(n) tile.)
    uint64_t *p_part = s_full + NSBUF;
    uint64_t *o_final = p_part + NSBUF * P_PARTS;
    uint64_t *drain = o_final + 1;
    uint64_t *pv_buf = drain + 1;          // [S buffer]: P.V of the tile in that buffer done
    uint64_t *m_ready = pv_buf + NSBUF;    // [tile parity][warp % 4]: row max after tile n published
    uint64_t *epi = m_ready + 8;           // [warp % 4]: both warps of a row pair posted (l, m)
    uint64_t *epi_done = epi + 4;          // [warp % 4]: both warps of a row pair have read O
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi_done + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint32_t *issued = tmem_slot + 2;      // K/V loads this CTA issued (CLUSTER exit protocol)

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t crank = CLUSTER ? cluster_ctarank() : 0u;  // this CTA's rank in its cluster

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NSTAGE; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_full[NSTAGE + s], 1);
            mbar_init(&kv_empty[s], CLUSTER ? 2 : 1);  // with CLUSTER: this CTA's release and the partner's
        }
        for (int b = 0; b < NSBUF; b++) mbar_init(&s_full[b], 1);
        for (int q = 0; q < NSBUF * P_PARTS; q++) mbar_init(&p_part[q], BM);
        mbar_init(o_final, 1);
        mbar_init(drain, 2);  // one commit per MMA issuer
        for (int b = 0; b < NSBUF; b++) mbar_init(&pv_buf[b], 1);
        for (int q = 0; q < 8; q++) mbar_init(&m_ready[q], 32);
        for (int q = 0; q < 4; q++) {
            mbar_init(&epi[q], 64);
            mbar_init(&epi_done[q], 64);
        }
        *abort_flag = 0;
        *issued = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    // with CLUSTER the partner's barriers must be initialised before any remote arrival or multicast
    if constexpr (CLUSTER) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{p.wait_limit_ns, p.err, abort_flag};
    const long u0 = (long)blockIdx.x * p.group, u1 = u0 + p.group;

    if (warp >= 8) {
        regs_decrease<REGS_CONTROL>();
        if (warp == 8) {
            // -------------------------------------------------- TMA producer
            // The whole warp runs the loop and waits; one elected lane arms the
            // barriers and issues the copies.
            const bool leader = elect_one();
            if (leader) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
                prefetch_tmap(&tm_jk);
                prefetch_tmap(&tm_jv);
            }
            uint32_t kv_idx = 0;  // K/V tile loads issued so far
            uint32_t uc = 0;      // units started by this CTA
            bool ok = true;
            for (long u = u0; u < u1 && ok; u++, uc++) {
                const Unit un = decode_unit(p, u);
                const TileRange tr = chunk_tiles(p, un.c);
                if (uc == 0 && leader) {  // the CTA's Q tile, once
                    mbar_arrive_expect_tx(q_full, QK8 ? PANEL : TILE);
                    for (int half = 0; half < (QK8 ? 1 : 2); half++)
                        tma_load_4d(smem + SMEM_Q + half * PANEL, &tm_q, q_full, half * 64, un.h, un.q0, un.b);
                }
                auto load = [&](int kv, int j) -> bool {  // kv 0: K_j, 1: V_j
                    int map, row, valid;
                    tr.at(j, map, row, valid);
                    const uint32_t slot = kv_idx % NSTAGE;
                    if (!mbar_wait_w(&kv_empty[slot], ((kv_idx / NSTAGE) & 1) ^ 1, w)) return false;
                    const CUtensorMap *tm = kv == 0 ? (map == 0 ? &tm_k : &tm_jk) : (map == 0 ? &tm_v : &tm_jv);
                    const bool one_panel = QK8 && kv == 0;  // an e4m3 K tile is one 16 KB panel
                    if (leader) {
                        uint8_t *dst = smem + SMEM_KV + slot * TILE;
                        if constexpr (CLUSTER) {
                            // arm this CTA's barriers for both panels of the load, then
                            // send this CTA's panel to both CTAs
                            uint64_t *bar = &kv_full[crank * NSTAGE + slot];
                            mbar_arrive_expect_tx(&kv_full[slot], PANEL);
                            mbar_arrive_expect_tx(&kv_full[NSTAGE + slot], PANEL);
                            tma_load_4d_multicast(dst + crank * PANEL, tm, bar, (int)crank * 64, un.h, row, un.b,
                                                  (uint16_t)0x3);
                        } else {
                            mbar_arrive_expect_tx(&kv_full[slot], one_panel ? PANEL : TILE);
                            tma_load_4d(dst, tm, &kv_full[slot], 0, un.h, row, un.b);
                            if (!one_panel) tma_load_4d(dst + PANEL, tm, &kv_full[slot], 64, un.h, row, un.b);
                        }
                    }
                    kv_idx++;
                    return true;
                };
                // K_0 .. K_{A-1}, then V_j K_{j+A}: the order k_load / v_load describe
                const int T = tr.T;
                for (int t = 0; t < KAHEAD && t < T && ok; t++) ok = load(0, t);
                for (int j = 0; j < T && ok; j++) ok = load(1, j) && (j + KAHEAD >= T || load(0, j + KAHEAD));
            }
            // let every copy issued into shared memory land before the CTA can exit
            // (with CLUSTER the K/V copies are waited for after the first cluster barrier)
            if (uc > 0) mbar_drain(q_full, 0, tc::DRAIN_NS);
            if constexpr (CLUSTER) {
                if (leader) *issued = kv_idx;
            } else {
                for (uint32_t idx = kv_idx > NSTAGE ? kv_idx - NSTAGE : 0; idx < kv_idx; idx++)
                    mbar_drain(&kv_full[idx % NSTAGE], (idx / NSTAGE) & 1, tc::DRAIN_NS);
            }
        } else if (warp == 9 || warp == 10) {
            // ------------------------------------------------- MMA issuers
            // Warp 9 issues every S(n) = Q K_n^T, warp 10 every O += P(n).V_n: one
            // issuer would share its sub-partition's issue slots with two softmax
            // warps and feed the tensor pipe too slowly.  Each issuer is a whole,
            // converged warp: all lanes wait and compute descriptors, one elected
            // lane issues the MMAs and commits (the _w forms).  K/V tile n counts
            // over the CTA's units.  S(n) goes into buffer n % 3, which held P(n-3):
            // it waits for pv_buf[n % 3], committed after the P.V of tile n-3, so
            // it never overwrites a P still to be read.  P(n).V waits for the
            // parts of P(n); pv_buf[n % 3] follows it.
            const uint32_t idesc_qk = p.idesc_qk;
            const uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
            const uint32_t sQ = smem_u32(smem + SMEM_Q), sKV = smem_u32(smem + SMEM_KV);
            const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);      // Q / K: K-major, SBO 1024
            const uint64_t dv0 = smem_desc_sw128(sKV, PANEL, 1024);  // V: MN-major, LBO = panel stride
            uint32_t kv_idx = 0;  // K/V loads consumed before this unit
            uint32_t tile = 0;    // K/V tiles of earlier units
            uint32_t uc = 0;
            bool ok = true;
            if (warp == 9) {
                // This warp also frees V(n-3)'s ring slot: it waits for that tile's P.V
                // anyway (pv_buf) before S(n), so the P.V thread needs no commit for it.
                uint32_t vslot[4] = {0, 0, 0, 0};  // ring slot of V(m) at m % 4
                for (long u = u0; u < u1 && ok; u++, uc++) {
                    const int T = chunk_tiles(p, decode_unit(p, u).c).T;
                    ok = uc > 0 || mbar_wait_w(q_full, 0, w);
                    for (int t = 0; t < T && ok; t++) {
                        const uint32_t n = tile + t;
                        const uint32_t kidx = kv_idx + k_load(t, T);
                        vslot[n % 4] = (kv_idx + v_load(t, T)) % NSTAGE;
                        if (n >= NSBUF) {  // before waiting for K(n): the slot before K(n) held V(n-4)
                            if (!(ok = mbar_wait_w(&pv_buf[n % NSBUF], (n / NSBUF - 1) & 1, w))) break;
                            if (lane == 0) {  // V(n-3) read by its P.V
                                uint64_t *e = &kv_empty[vslot[(n - NSBUF) % 4]];
                                mbar_arrive(e);
                                if constexpr (CLUSTER) mbar_arrive_cluster(cluster_addr(e, crank ^ 1u));
                            }
                        }
                        if (!(ok = mbar_wait_w(&kv_full[kidx % NSTAGE], (kidx / NSTAGE) & 1, w))) break;
                        if constexpr (CLUSTER)  // the partner's panel
                            if (!(ok = mbar_wait_w(&kv_full[NSTAGE + kidx % NSTAGE], (kidx / NSTAGE) & 1, w))) break;
                        tc_fence_after();
                        const uint64_t kb = dq0 + ((uint64_t)(SMEM_KV - SMEM_Q + (kidx % NSTAGE) * TILE) >> 4);
                        if constexpr (QK8) {  // 32 head dims (32 bytes of each row) per MMA
#pragma unroll
                            for (int kk = 0; kk < D / 32; kk++) {
                                const uint64_t off = (uint64_t)(kk * 32) >> 4;
                                mma_ss_f8_w(tmem + (n % NSBUF) * BN, dq0 + off, kb + off, idesc_qk, kk > 0);
                            }
                        } else {  // 16 head dims per MMA, 4 per 64-dim panel
#pragma unroll
                            for (int kk = 0; kk < D / 16; kk++) {
                                const uint64_t off = (uint64_t)((kk >> 2) * PANEL + (kk & 3) * 32) >> 4;
                                mma_ss_w(tmem + (n % NSBUF) * BN, dq0 + off, kb + off, idesc_qk, kk > 0);
                            }
                        }
                        tc_commit_w(&s_full[n % NSBUF]);  // K(n)'s slot is freed by the softmax, which sees S(n)
                    }
                    kv_idx += 2 * T;
                    tile += T;
                }
            } else {
                for (long u = u0; u < u1 && ok; u++, uc++) {
                    const int T = chunk_tiles(p, decode_unit(p, u).c).T;
                    const bool carry = p.merge && uc > 0;      // O accumulates over the previous chunks
                    const bool last = !p.merge || u + 1 == u1;  // this chunk's O goes to the epilogue
                    for (int j = 0; j < T && ok; j++) {
                        const uint32_t n = tile + j;
                        const uint32_t vidx = kv_idx + v_load(j, T);  // V_j
                        // the slot's previous load, K(n-1), has landed: P(n-1).V was issued
                        if (!(ok = mbar_wait_w(&kv_full[vidx % NSTAGE], (vidx / NSTAGE) & 1, w))) break;
                        if constexpr (CLUSTER)
                            if (!(ok = mbar_wait_w(&kv_full[NSTAGE + vidx % NSTAGE], (vidx / NSTAGE) & 1, w))) break;
                        // P(n) (bf16, keys in order) sits over the first BN/2 columns of its buffer;
                        // each part's P.V starts as soon as the softmax has published that part
                        const uint64_t vb = dv0 + ((uint64_t)((vidx % NSTAGE) * TILE) >> 4);
                        const uint32_t pb = tmem + (n % NSBUF) * BN;
                        for (int q = 0; q < P_PARTS && ok; q++) {
                            if (!(ok = mbar_wait_w(&p_part[(n % NSBUF) * P_PARTS + q], (n / NSBUF) & 1, w))) break;
                            tc_fence_after();
#pragma unroll
                            for (int kk = q * (KP / 16); kk < (q + 1) * (KP / 16); kk++)
                                mma_ts_w(tmem + O_COL, pb + kk * 8, vb + ((uint64_t)(kk * 16 * 128) >> 4), idesc_pv,
                                       (carry || j > 0 || kk > 0) ? 1u : 0u);
                        }
                        if (!ok) break;
                        tc_commit_w(&pv_buf[n % NSBUF]);
                        if (j + 1 == T && last) tc_commit_w(o_final);
                    }
                    kv_idx += 2 * T;
                    tile += T;
                }
            }
            // every MMA issued so far must complete before tensor memory is freed
            // (the drain barrier counts one commit per issuer)
            tc_commit_w(drain);
            mbar_drain(drain, 0, tc::DRAIN_NS);
        }
        __syncwarp();
    } else {
        regs_increase<REGS_SOFTMAX>();
        // ------------------------------------ softmax / epilogue (warpgroup hf)
        // Warpgroup hf takes the K/V tiles n with n % 2 == hf, whole rows (thread =
        // row = TMEM lane; warps w and w + 4 reach the same lanes), so that each
        // group has two tiles' time for one tile's softmax.  The groups share the
        // row's running max: tile n's owner waits for the max after tile n-1
        // (m_ready), takes the new max, posts it and only then computes P(n).  The
        // max moves, and O is rescaled in tensor memory, only when the tile max
        // exceeds it by 2^8 (a lazy rescale: the same stale max scales numerator
        // and denominator).  Each group keeps the row sum of its own tiles,
        // expressed in the max it last saw; the epilogue combines the two.
        const int hf = warp / 4, wq = warp % 4;
        const int r = threadIdx.x % BM;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * wq) << 16);
        const uint32_t tO = lane_base + O_COL;
        float *xm = reinterpret_cast<float *>(smem + SMEM_XCH);  // [row]: max after the latest tile
        float *xe = xm + BM;                                      // [group][row][l, m]
        const float sl2 = p.scale_log2;
        uint32_t tile = 0, uc = 0, n_epi = 0;
        uint32_t kv_idx = 0;      // K/V loads of earlier units
        bool ok = true;
        float m_run = -INFINITY;  // the row max in force after the latest tile of this unit
        float m_own = -INFINITY;  // the max l_own is expressed in
        float l_own = 0.f;        // row sum over this group's tiles
        for (long u = u0; u < u1 && ok; u++, uc++) {
            const Unit un = decode_unit(p, u);
            const TileRange tr = chunk_tiles(p, un.c);
            const int T = tr.T;
            const bool carry = p.merge && uc > 0;      // (m, l, O) of the previous chunks carry over
            const bool last = !p.merge || u + 1 == u1;
            if (!carry) m_run = -INFINITY, m_own = -INFINITY, l_own = 0.f;
            if constexpr (BOUNDED) {
                const long grow = (long)un.q0 + r;
                m_run = grow < p.Sq ? p.row_bound[((long)un.b * p.H + un.h) * p.Sq + grow] * 1.4426950408889634f
                                    : 0.f;
                m_own = m_run;
            }
            for (int j = 0; j < T; j++) {
                const uint32_t n = tile + j;
                if ((int)(n & 1) != hf) continue;  // the other group's tile
                int map, row, valid;
                tr.at(j, map, row, valid);
                const uint32_t tS = lane_base + (n % NSBUF) * BN;
                if (!mbar_wait(&s_full[n % NSBUF], (n / NSBUF) & 1, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S(n) is complete: K(n)'s ring slot is free
                if (r == 0) {
                    uint64_t *e = &kv_empty[(kv_idx + k_load(j, T)) % NSTAGE];
                    mbar_arrive(e);
                    if constexpr (CLUSTER) mbar_arrive_cluster(cluster_addr(e, crank ^ 1u));
                }
                if constexpr (!BOUNDED) {
                    // the max after tile n-1 (posted by the other group early in its
                    // tile), every phase waited in turn
                    if (n > 0) {
                        if (!mbar_wait(&m_ready[((n - 1) & 1) * 4 + wq], ((n - 1) >> 1) & 1, w)) {
                            ok = false;
                            break;
                        }
                        if (j > 0 || carry) m_run = xm[r];
                    }
                }
                uint32_t s[BN];
#pragma unroll
                for (int cc = 0; cc < BN / 32; cc++)
                    tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
                tmem_ld_wait();
                if (valid < BN) {  // ragged tile end (warp-uniform): keys past the segment get -inf
#pragma unroll
                    for (int k = 0; k < BN; k++)
                        if (k >= valid) s[k] = 0xff800000u;
                }
                bool rescale = false;  // warp-uniform
                float alpha = 1.f;
                if constexpr (!BOUNDED) {
                    float mc[4];
#pragma unroll
                    for (int c4 = 0; c4 < 4; c4++) {
                        const uint32_t *x = &s[c4 * 32];
                        float m = fmax3(__uint_as_float(x[0]), __uint_as_float(x[1]), __uint_as_float(x[2]));
#pragma unroll
                        for (int k = 3; k < 31; k += 2) m = fmax3(m, __uint_as_float(x[k]), __uint_as_float(x[k + 1]));
                        mc[c4] = fmaxf(m, __uint_as_float(x[31]));
                    }
                    const float mt = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * sl2;
                    bool need = false;
                    if (j == 0 && !carry) m_run = mt;
                    else need = mt > m_run + tc::RESCALE_THRESHOLD;
                    if (__any_sync(0xffffffffu, need)) {
                        rescale = true;
                        if (need) {
                            alpha = ex2(m_run - mt);
                            m_run = mt;
                        }
                    }
                    xm[r] = m_run;
                    mbar_arrive(&m_ready[(n & 1) * 4 + wq]);
                    if (m_own != m_run) {
                        l_own = l_own > 0.f ? l_own * ex2(m_own - m_run) : 0.f;
                        m_own = m_run;
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
                        // O holds P.V of tiles < n once P(n-1).V is done; rescale it before P(n).V
                        if (!mbar_wait(&pv_buf[(n - 1) % NSBUF], ((n - 1) / NSBUF) & 1, w)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
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
                    mbar_arrive(&p_part[(n % NSBUF) * P_PARTS + q]);
                }
                if (!ok) break;
                float a0, a1, b0, b1;
                f2_split(fadd2(acc[0], acc[1]), a0, a1);
                f2_split(fadd2(acc[2], acc[3]), b0, b1);
                l_own += (a0 + a1) + (b0 + b1);
            }
            if (!ok) break;
            if (!last) {  // the group's partial is written after its last chunk
                tile += T;
                kv_idx += 2 * T;
                continue;
            }
            // epilogue: the two groups combine their row sums, each writes half of O's
            // columns; both have read O before either publishes the next unit's P
            if (!mbar_wait(o_final, n_epi & 1, w)) {
                ok = false;
                break;
            }
            // one buffer serves every unit: both groups have read it (epi_done) before either
            // writes the next unit's (l, m)
            float *xs = xe;
            xs[(hf * BM + r) * 2] = l_own;
            xs[(hf * BM + r) * 2 + 1] = m_own;
            mbar_arrive(&epi[wq]);
            if (!mbar_wait(&epi[wq], n_epi & 1, w)) {
                ok = false;
                break;
            }
            const float l_oth = xs[((hf ^ 1) * BM + r) * 2], m_oth = xs[((hf ^ 1) * BM + r) * 2 + 1];
            const float m_fin = fmaxf(m_own, m_oth);  // the max O is expressed in
            const float l_tot = (l_own > 0.f ? l_own * ex2(m_own - m_fin) : 0.f) +
                                (l_oth > 0.f ? l_oth * ex2(m_oth - m_fin) : 0.f);
            const long pc = p.merge ? un.c / p.group : un.c;  // index of the partial written
            const long grow = (long)un.q0 + r;
            const bool live = grow < p.Sq;
            tc_fence_after();
            if constexpr (BOUNDED) {
                if (live && !(l_tot > 0.f)) atomicCAS(p.err, DEV_OK, DEV_RANGE);  // all terms underflowed
            }
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const long obase = (((long)un.b * p.Sq + (live ? grow : 0)) * p.H + un.h) * D + hf * (D / 2);
#pragma unroll
            for (int cc = 0; cc < D / 64; cc++) {
                uint32_t o[32];
                tmem_ld32(tO + hf * (D / 2) + cc * 32, o);
                tmem_ld_wait();
                if (live) {
                    if (p.out_f32) {
                        // streaming stores: the partials are read once, by the merge
                        float *dst = static_cast<float *>(p.out) + (long long)pc * p.o_stride + obase + cc * 32;
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
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
            if (live && p.lse && hf == 0)
                p.lse[(long long)pc * p.l_stride + ((long)un.b * p.H + un.h) * p.Sq + grow] =
                    (m_fin + log2f(l_tot)) * 0.69314718055994531f;
            tc_fence_before();
            mbar_arrive(&epi_done[wq]);
            if (!mbar_wait(&epi_done[wq], n_epi & 1, w)) {
                ok = false;
                break;
            }
            n_epi++;
            tile += T;
            kv_idx += 2 * T;
        }
    }

    tc_fence_before();
    if constexpr (CLUSTER) {
        cluster_sync();  // neither CTA issues a copy or a remote arrival any more
        if (warp == 8) {
            // wait for the last load of each source CTA in each slot to land here
            // (earlier loads of a slot landed before it could be refilled).  This
            // CTA armed both panels of each load it issued; the partner, at most
            // one load a slot ahead (it refills a slot only after this CTA's
            // consumers released it), may have sent a panel this CTA never
            // armed: arm that phase now, so that it completes when the bytes land.
            const uint32_t mine = *issued, theirs = ld_cluster_u32(cluster_addr(issued, crank ^ 1u));
            for (uint32_t s = lane; s < (uint32_t)NSTAGE; s += 32) {
                if (mine > s) {
                    const uint32_t last = s + NSTAGE * ((mine - 1 - s) / NSTAGE);
                    mbar_drain(&kv_full[crank * NSTAGE + s], (last / NSTAGE) & 1, tc::DRAIN_NS);
                }
                if (theirs > s) {
                    const uint32_t last = s + NSTAGE * ((theirs - 1 - s) / NSTAGE);
                    uint64_t *bar = &kv_full[(crank ^ 1u) * NSTAGE + s];
                    if (last >= mine) mbar_arrive_expect_tx(bar, PANEL);
                    mbar_drain(bar, (last / NSTAGE) & 1, tc::DRAIN_NS);
                }
            }
        }
        cluster_sync();  // no CTA leaves while a copy may still land in it
    } else {
        __syncthreads();
    }
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------- host

cudaError_t launch_attn_tc_single(const Geom &g, const void *q, const void *k, const void *v, const void *jk,
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
    // Clusters of two CTAs share every K/V tile (16-bit q/k).  The pair holds Q
    // tiles 2i and 2i+1, so an odd tile count gets one all-padding tile per
    // (batch, head, chunk group), worth it only when there are enough tiles.
    const long q_tiles = (g.Sq + tc::BM - 1) / tc::BM;
    const bool cluster = K6_KV_MULTICAST && !opt.qk8 && (q_tiles % 2 == 0 || q_tiles >= 16);
    auto kernel = opt.qk8   ? (opt.row_bound ? attn_tc_single_kernel<true, true, false>
                                             : attn_tc_single_kernel<false, true, false>)
                  : cluster ? (opt.row_bound ? attn_tc_single_kernel<true, false, true>
                                             : attn_tc_single_kernel<false, false, true>)
                            : (opt.row_bound ? attn_tc_single_kernel<true, false, false>
                                             : attn_tc_single_kernel<false, false, false>);
    cudaError_t attr_err = set_max_dynamic_smem((const void *)kernel, ts::SMEM_ALLOC);
    if (attr_err != cudaSuccess) return attr_err;
    TcParams p;
    p.S = g.S;
    p.Sq = g.Sq;
    p.Nv = g.Nv;
    p.Nj = g.Nj;
    p.H = g.H;
    p.n_chunks = n_chunks;
    p.q_tiles = (int)(cluster ? (q_tiles + 1) / 2 * 2 : q_tiles);  // rows >= Sq are masked
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
    p.units = (long)g.B * g.H * n_chunks * p.q_tiles;
    if (p.units == 0) return cudaSuccess;
    if (p.units >= (1L << 31)) {
        if (why) *why = "too many work units (batch x heads x chunks must stay below 2^31)";
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
    p.row_bound = opt.row_bound;
    const long grid = p.units / p.group;  // even with cluster: q_tiles is
    if (!cluster) {
        kernel<<<(unsigned)grid, ts::THREADS, ts::SMEM_ALLOC, st>>>(mq, mk, mv, mjk, mjv, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(ts::THREADS);
    cfg.dynamicSmemBytes = ts::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mjk, mjv, p);
}

}  // namespace k6
