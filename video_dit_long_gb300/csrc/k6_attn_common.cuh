// k6_attn_common.cuh -- launch parameters of the bf16 tensor-core attention
// kernel, the K/V tile range of a chunk of the joint sequence, and the mapping
// of work units to CTAs.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "k6_internal.h"

namespace k6 {

namespace tc {
constexpr int D = 128;
constexpr int BM = 128;                       // query rows per Q tile
constexpr int BN = 128;                       // keys per K/V tile
constexpr int PANEL = BM * 64 * 2;            // one 128-row x 64-dim bf16 panel: 16 KB
constexpr int TILE = 2 * PANEL;               // 32 KB
constexpr float RESCALE_THRESHOLD = 8.0f;     // log2 units: rescale when the max grows past 2^8
constexpr unsigned long long DRAIN_NS = 1000000000ull;
}  // namespace tc

struct TcParams {
    long S, Nv, Nj;                           // keys (video then joint)
    long Sq;                                  // query rows
    int H, n_chunks, q_tiles;                 // q_tiles: 128-row query tiles per (b, h)
    float scale_log2;                         // log2(e) / sqrt(d)
    void *out;                                // bf16 [B][S][H][d] or fp32 partials
    float *lse;
    int out_f32;
    long long o_stride, l_stride;             // elements between chunks
    unsigned long long wait_limit_ns;
    int *err;
    int strict_order;
    uint32_t idesc_qk;                        // instruction descriptor of Q.K^T (bf16 or fp16 operands)
    long units;                               // B * H * n_chunks * q_tiles work units
    int group;                                // chunks per CTA, sharing one load of Q (divides n_chunks)
    int merge;                                // 1: a CTA's group of chunks leaves one partial (index c / group)
    const float *row_bound;                   // constant-max softmax: bound per query row [B][H][Sq], or null
};

// K/V tile j of a chunk: which tensor map (0 video, 1 joint), first row, valid
// keys.  32-bit arithmetic: the host keeps S below 2^30 and the unit count
// below 2^31.
struct TileRange {
    int v_beg, v_end, j_beg, j_end;
    int Tv, T;
    __device__ void at(int j, int &map, int &row, int &valid) const {
        if (j < Tv) {
            map = 0;
            row = v_beg + j * tc::BN;
            valid = min(tc::BN, v_end - row);
        } else {
            map = 1;
            row = j_beg + (j - Tv) * tc::BN;
            valid = min(tc::BN, j_end - row);
        }
    }
};

__device__ __forceinline__ TileRange chunk_tiles(const TcParams &p, int c) {
    TileRange t;
    const int S = (int)p.S, Nv = (int)p.Nv;
    const int L = S / p.n_chunks;
    const int kb = c * L, ke = kb + L;
    t.v_beg = kb;
    t.v_end = ke < Nv ? ke : Nv;
    t.j_beg = (kb > Nv ? kb : Nv) - Nv;
    t.j_end = ke > Nv ? ke - Nv : 0;
    t.Tv = t.v_end > t.v_beg ? (t.v_end - t.v_beg + tc::BN - 1) / tc::BN : 0;
    const int Tj = t.j_end > t.j_beg ? (t.j_end - t.j_beg + tc::BN - 1) / tc::BN : 0;
    t.T = t.Tv + Tj;
    return t;
}

// Work unit u -> (b, h, chunk group, query tile, chunk within the group),
// the chunk within the group fastest: CTA x owns units [x*group, (x+1)*group),
// one Q tile over `group` consecutive chunks.  Across CTAs the query tile
// varies fastest, so the CTAs running at the same time walk through the
// same chunks and share their K/V in L2.
struct Unit {
    int b, h, c, q0;
};
__device__ __forceinline__ Unit decode_unit(const TcParams &p, long unit) {
    Unit r;
    uint32_t u = (uint32_t)unit;
    const uint32_t g = u % (uint32_t)p.group;
    u /= (uint32_t)p.group;
    const uint32_t qp = u % (uint32_t)p.q_tiles;
    u /= (uint32_t)p.q_tiles;
    const uint32_t groups = (uint32_t)(p.n_chunks / p.group);
    const uint32_t cg = u % groups;
    u /= groups;
    r.c = (int)(cg * p.group + g);
    r.h = (int)(u % (uint32_t)p.H);
    r.b = (int)(u / (uint32_t)p.H);
    r.q0 = (int)qp * tc::BM;
    return r;
}

}  // namespace k6
