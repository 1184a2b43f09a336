// k6_rope.cu -- rotary embedding of Q and K for the joint video/text sequence.
//
// "Context Parallelism in vLLM Omni Neuron", sections "Self-Attention with
// Context Parallelism" (`apply_rotary_emb_wan` on query and key after QK-norm,
// before attention) and "Positional Embedding Handling" (per-token cos/sin
// tables, sliced by token range).  The pages print no formula; this library
// reads it as: each axis (t, h, w) owns a contiguous segment of axis_dim[a]
// head dims, in that order; pair i of the segment, dims (2i, 2i+1), turns by
// pos_a * theta^(-2i/axis_dim[a]) as the complex product (x + iy) e^{i angle};
// joint tokens are unrotated, or (joint_rope) turn over the full head dim by
// their 0-based joint index.
//
// Tables are factorised per axis (grid_t + grid_h + grid_w rows instead of
// one row per token), fp32 (cos, sin), built once per handle in fp64.
// The rotation kernel is HBM-bound: one 16-byte load and one 16-byte store
// per 8 bf16 (or 4 f32) elements; Q, K and joint K are rotated in one launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "k6_device.cuh"
#include "k6_internal.h"

namespace k6 {

RopeLayout rope_layout(const Geom &g) {
    RopeLayout L;
    L.off[0] = 0;
    L.off[1] = L.off[0] + (long)g.grid_t * (g.axis_dim[0] / 2);
    L.off[2] = L.off[1] + (long)g.grid_h * (g.axis_dim[1] / 2);
    L.off[3] = L.off[2] + (long)g.grid_w * (g.axis_dim[2] / 2);
    L.total = L.off[3] + (g.joint_rope ? g.Nj * (g.d / 2) : 0);
    return L;
}

struct TableArgs {
    long off[4];
    long total;
    int half[4];    // pairs per row: axis_dim[a]/2, and d/2 for the joint table
    int dims[4];    // rotating dims of each table: axis_dim[a], d
    double theta;
};

__global__ void rope_table_kernel(TableArgs a, float2 *tab) {
    long i = blockIdx.x * (long)blockDim.x + threadIdx.x;
    if (i >= a.total) return;
    int t = 0;
    while (t < 3 && i >= a.off[t + 1]) t++;
    long local = i - a.off[t];
    long pos = local / a.half[t];
    int pair = (int)(local % a.half[t]);
    double omega = pow(a.theta, -2.0 * pair / a.dims[t]);
    double s, c;
    sincos((double)pos * omega, &s, &c);
    tab[i] = make_float2((float)c, (float)s);
}

cudaError_t launch_rope_tables(const Geom &g, double theta, float2 *tables, cudaStream_t st) {
    RopeLayout L = rope_layout(g);
    TableArgs a;
    for (int t = 0; t < 4; t++) a.off[t] = L.off[t];
    a.total = L.total;
    for (int t = 0; t < 3; t++) {
        a.half[t] = g.axis_dim[t] / 2 > 0 ? g.axis_dim[t] / 2 : 1;
        a.dims[t] = g.axis_dim[t] > 0 ? g.axis_dim[t] : 1;
    }
    a.half[3] = g.d / 2;
    a.dims[3] = g.d;
    a.theta = theta;
    if (L.total == 0) return cudaSuccess;
    int threads = 256;
    long blocks = (L.total + threads - 1) / threads;
    rope_table_kernel<<<(unsigned)blocks, threads, 0, st>>>(a, tables);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ rotate

struct RopeArgs {
    int *err;            // device error word (range check of fp16 output)
    const void *src[3];
    void *dst[3];
    long tokens[3];      // B*S, B*Nv, B*Nj
    long seq[3];         // S, Nv, Nj  (tokens per batch)
    long Nv;
    int H, d;
    int grid_h, grid_w;
    int seg1, seg2;      // first pair index of the h and w segments
    int joint_rope;
    long off[4];         // table offsets (float2 entries)
    int half[3];         // pairs per axis row
    // QK-norm weights, fp32 [H*d]: [tensor][0 = video rows, 1 = joint rows]
    // (tensor 0 = q, 1 = k, 2 = joint_k); all null = no norm
    const float *norm_w[3][2];
    float eps;
};

// (cos, sin) of pair `i` for a token with video position (t, h, w), or joint
// index j (j >= 0 means joint).
__device__ __forceinline__ float2 rope_cs(const RopeArgs &a, const float2 *tab, int i, int t, int h, int w,
                                          long j) {
    if (j >= 0) {
        if (!a.joint_rope) return make_float2(1.f, 0.f);
        return tab[a.off[3] + j * (a.d / 2) + i];
    }
    if (i < a.seg1) return tab[a.off[0] + (long)t * a.half[0] + i];
    if (i < a.seg2) return tab[a.off[1] + (long)h * a.half[1] + (i - a.seg1)];
    return tab[a.off[2] + (long)w * a.half[2] + (i - a.seg2)];
}

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int kPairs = 4;
    __device__ static void load(const void *p, float (&x)[8]) {
        uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
        for (int k = 0; k < 4; k++) {
            float2 f = __bfloat1622float2(b[k]);
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    }
    __device__ static void store(void *p, const float (&x)[8]) {
        uint4 u;
        __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&u);
        for (int k = 0; k < 4; k++) b[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};
template <>
struct Vec<__half> {
    static constexpr int kPairs = 4;
    __device__ static void store(void *p, const float (&x)[8]) {
        uint4 u;
        __half2 *b = reinterpret_cast<__half2 *>(&u);
        for (int k = 0; k < 4; k++) b[k] = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};
template <>
struct Vec<float> {
    static constexpr int kPairs = 2;
    __device__ static void load(const void *p, float (&x)[8]) {
        float4 u = *reinterpret_cast<const float4 *>(p);
        x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w;
    }
    __device__ static void store(void *p, const float (&x)[8]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

// One warp per token: its H*d elements are contiguous, the token's position
// (and so its rotation angles) is uniform across the warp, and each lane
// moves up to 4 16-byte vectors per pass with all loads issued before any
// store, so that enough bytes are in flight for HBM.
// With NORM, each token row of H*d values is first RMS-normalised
// (x * rsqrt(mean(x^2) + eps) * w, fp32): one pass sums the squares (warp
// reduction), the second pass re-reads the row (an L2 hit) and normalises.
// Token `tok` of the concatenation (q rows, k rows, joint_k rows): which
// tensor, its row there, and its rotary position: video grid (t, h, w), or
// joint index j >= 0.  32-bit arithmetic: the host keeps B*S*H below 2^31.
struct TokenPos {
    int which;
    unsigned local;
    int t, h, w;
    long j;
};
__device__ __forceinline__ TokenPos token_pos(const RopeArgs &a, long tok) {
    TokenPos p;
    p.which = 0;
    p.local = (unsigned)tok;
    while (p.which < 2 && p.local >= (unsigned)a.tokens[p.which]) {
        p.local -= (unsigned)a.tokens[p.which];
        p.which++;
    }
    const unsigned n = p.local % (unsigned)a.seq[p.which];  // token index within its sequence
    p.j = -1;
    if (p.which == 2) p.j = n;
    else if (n >= (unsigned)a.Nv) p.j = n - (unsigned)a.Nv;
    p.t = p.h = p.w = 0;
    if (p.j < 0) {
        const unsigned gw = (unsigned)a.grid_w, gh = (unsigned)a.grid_h;
        const unsigned nw = n / gw;
        p.w = (int)(n - nw * gw);
        p.t = (int)(nw / gh);
        p.h = (int)(nw - (unsigned)p.t * gh);
    }
    return p;
}

// A lane's vectors are v = lane + 32 u, and a head row holds d / (2 kPairs)
// vectors, a divisor of 32 for every supported d: so a lane always rotates the
// same kPairs pairs of every head, and reads their cos/sin once per token.
template <typename T, typename Tout, bool NORM>
__global__ void __launch_bounds__(256) rope_kernel(RopeArgs a, const float2 *__restrict__ tab) {
    constexpr int kPairs = Vec<T>::kPairs;
    constexpr int kUnroll = 6;
    static_assert(sizeof(T) == sizeof(Tout), "rotation keeps the element size");
    const long total = a.tokens[0] + a.tokens[1] + a.tokens[2];
    const int vecs_per_token = a.H * a.d / (2 * kPairs);
    const int vecs_per_head = a.d / (2 * kPairs);
    const int lane = threadIdx.x & 31;
    const long warp0 = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    for (long tok = warp0; tok < total; tok += nwarps) {
        const TokenPos tp = token_pos(a, tok);
        const int which = tp.which, t = tp.t, h = tp.h, w = tp.w;
        const unsigned local = tp.local;
        const long j = tp.j;
        const char *src = static_cast<const char *>(a.src[which]) + (long)local * a.H * a.d * sizeof(T);
        char *dst = static_cast<char *>(a.dst[which]) + (long)local * a.H * a.d * sizeof(T);
        bool bad = false;
        float inv_rms = 1.f;
        const float *wrow = nullptr;
        if constexpr (NORM) {
            wrow = a.norm_w[which][j >= 0 ? 1 : 0];
            float ss = 0.f;
            for (int v = lane; v < vecs_per_token; v += 32) {
                float x[8];
                Vec<T>::load(src + (long)v * 16, x);
#pragma unroll
                for (int k = 0; k < 2 * kPairs; k++) ss = fmaf(x[k], x[k], ss);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            inv_rms = rsqrtf(ss / (float)(a.H * a.d) + a.eps);
        }
        const int pair0 = (lane % vecs_per_head) * kPairs;
        float2 cs[kPairs];
#pragma unroll
        for (int k = 0; k < kPairs; k++) cs[k] = rope_cs(a, tab, pair0 + k, t, h, w, j);
        for (int base = 0; base < vecs_per_token; base += 32 * kUnroll) {
            float x[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                const int v = base + u * 32 + lane;
                if (v < vecs_per_token) Vec<T>::load(src + (long)v * 16, x[u]);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                const int v = base + u * 32 + lane;
                if (v >= vecs_per_token) continue;
                if constexpr (NORM) {
                    const float *wv = wrow + v * 2 * kPairs;
#pragma unroll
                    for (int k = 0; k < 2 * kPairs; k++) x[u][k] *= inv_rms * __ldg(wv + k);
                }
#pragma unroll
                for (int k = 0; k < kPairs; k++) {
                    const float xr = x[u][2 * k], xi = x[u][2 * k + 1];
                    x[u][2 * k] = xr * cs[k].x - xi * cs[k].y;
                    x[u][2 * k + 1] = xr * cs[k].y + xi * cs[k].x;
                }
                if constexpr (!std::is_same<T, Tout>::value) {
#pragma unroll
                    for (int k = 0; k < 2 * kPairs; k++) bad |= !(fabsf(x[u][k]) < 65520.f);  // a finite half
                }
                Vec<Tout>::store(dst + (long)v * 16, x[u]);
            }
        }
        if (bad) atomicCAS(a.err, DEV_OK, DEV_RANGE);
    }
}

// Short token rows (a head-partitioned layout keeps H/P heads per token, e.g.
// 3 x 128 elements): a group of `gl` lanes (16, or 32 when a head holds 32
// vectors) owns whole rows; each lane decodes its rows' positions and reads
// its 4 cos/sin once per row, then moves `vpl` vectors of each of `rpg` rows,
// kUnroll 16-byte loads in flight.  Rotation only (no QK-norm, whose statistic
// needs the full row).  A lane's vectors are sub + gl*u of a row, and a head a
// divisor of gl vectors, so the lane stays on the same kPairs pairs of every
// head.
template <typename T, typename Tout>
__global__ void __launch_bounds__(256) rope_short_kernel(RopeArgs a, const float2 *__restrict__ tab, int gl, int vpl,
                                                         int rpg) {
    constexpr int kPairs = Vec<T>::kPairs;
    constexpr int kUnroll = 6;
    constexpr int kRows = kUnroll;             // rows per group pass at most (vpl >= 1)
    const long total = a.tokens[0] + a.tokens[1] + a.tokens[2];
    const int vpt = a.H * a.d / (2 * kPairs);  // vectors per token row
    const int vph = a.d / (2 * kPairs);        // vectors per head
    const int lane = threadIdx.x & 31;
    const int sub = lane % gl, grp = lane / gl, groups = 32 / gl;
    const int pair0 = (sub % vph) * kPairs;
    const long warp0 = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const long per_pass = (long)groups * rpg;  // rows per warp pass
    bool bad = false;
    for (long row0 = warp0 * per_pass + (long)grp * rpg; row0 < total; row0 += nwarps * per_pass) {
        float x[kUnroll][8];
        float2 cs[kRows][kPairs];
        const char *src[kRows];
        char *dst[kRows];
#pragma unroll
        for (int r = 0; r < kRows; r++) {
            src[r] = nullptr;
            if (r < rpg && row0 + r < total) {
                const TokenPos tp = token_pos(a, row0 + r);
                src[r] = static_cast<const char *>(a.src[tp.which]) + (long)tp.local * vpt * 16;
                dst[r] = static_cast<char *>(a.dst[tp.which]) + (long)tp.local * vpt * 16;
#pragma unroll
                for (int k = 0; k < kPairs; k++) cs[r][k] = rope_cs(a, tab, pair0 + k, tp.t, tp.h, tp.w, tp.j);
            }
        }
        // element e = r * vpl + i: row r, the lane's vector sub + gl * i of that row
#pragma unroll
        for (int e = 0; e < kUnroll; e++) {
            const int r = e / vpl, v = sub + gl * (e - r * vpl);
            if (r < rpg && src[r] && v < vpt) Vec<T>::load(src[r] + (long)v * 16, x[e]);
        }
#pragma unroll
        for (int e = 0; e < kUnroll; e++) {
            const int r = e / vpl, v = sub + gl * (e - r * vpl);
            if (!(r < rpg && src[r] && v < vpt)) continue;
#pragma unroll
            for (int k = 0; k < kPairs; k++) {
                const float xr = x[e][2 * k], xi = x[e][2 * k + 1];
                x[e][2 * k] = xr * cs[r][k].x - xi * cs[r][k].y;
                x[e][2 * k + 1] = xr * cs[r][k].y + xi * cs[r][k].x;
            }
            if constexpr (!std::is_same<T, Tout>::value) {
#pragma unroll
                for (int k = 0; k < 2 * kPairs; k++) bad |= !(fabsf(x[e][k]) < 65520.f);  // a finite half
            }
            Vec<Tout>::store(dst[r] + (long)v * 16, x[e]);
        }
    }
    if (bad) atomicCAS(a.err, DEV_OK, DEV_RANGE);
}

// ------------------------------------------------ rotary + head split, fused
//
// The Ulysses prologue of one attention layer in one pass: rotary embeddings of
// q, k and joint_k and the sequence->head relayout of q, k, joint_k, v and
// joint_v ("Context Parallelism in vLLM Omni Neuron", "Self-Attention with
// Context Parallelism": rotary on the local tokens before attention; xDiT PR
// #586, USP dispatch listing, `_ft_c_input_all_to_all`).  Source rows are
// BSHD bf16 token rows of H*128 elements (H*16 16-byte vectors); vector v of
// a row belongs to head v/16, i.e. to head group p = v/(16*Hl), and lands in
//   dst[p][b][n][v - 16*Hl*p]   (16-byte vectors; layout [P][B][rows][Hl][128]).
// One warp per row: every load of the row is issued before its first store
// (the outputs never alias the inputs), 12 vectors per lane for H = 24.  The
// lane's 16-byte vectors always hold the same 4 pairs of their heads (16
// vectors per head divide 32), so their cos/sin are read once per row.
struct SplitArgs {
    RopeArgs r;              // rotary tables and positions (tensors 0..2 = q, k, joint_k)
    const void *src[5];      // q, k, joint_k, v, joint_v
    void *dst[5];
    long count[5];           // rows per tensor: B*S, B*Nv, B*Nj, B*Nv, B*Nj
    long seq[5];             // rows per batch of each tensor
    int B, P, Hl;
};

template <typename TQK>
__global__ void __launch_bounds__(256) rope_split_kernel(SplitArgs a, const float2 *__restrict__ tab) {
    constexpr int kU = 12;                        // vectors per lane in flight
    const int vpt = a.r.H * 16;                   // 16-byte vectors per row
    const int vpp = a.Hl * 16;                    // vectors per head group
    const long total = a.count[0] + a.count[1] + a.count[2] + a.count[3] + a.count[4];
    const int lane = threadIdx.x & 31;
    const long warp0 = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const int pair0 = (lane & 15) * 4;
    bool bad = false;
    for (long row = warp0; row < total; row += nwarps) {
        int which = 0;
        long local = row;
        while (which < 4 && local >= a.count[which]) {
            local -= a.count[which];
            which++;
        }
        const bool rot = which < 3;
        float2 cs[4] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f), make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
        if (rot) {
            // the row's position: token_pos walks q, k, joint_k in that order
            long tok = local;
            for (int t = 0; t < which; t++) tok += a.r.tokens[t];
            const TokenPos tp = token_pos(a.r, tok);
#pragma unroll
            for (int k = 0; k < 4; k++) cs[k] = rope_cs(a.r, tab, pair0 + k, tp.t, tp.h, tp.w, tp.j);
        }
        const unsigned seq = (unsigned)a.seq[which];  // 32-bit: the host keeps B*S*H below 2^31
        const unsigned b = (unsigned)local / seq, n = (unsigned)local - b * seq;
        const uint4 *src = static_cast<const uint4 *>(a.src[which]) + local * vpt;
        char *dst = static_cast<char *>(a.dst[which]);
        for (int base = 0; base < vpt; base += 32 * kU) {
            uint4 x[kU];
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const int v = base + 32 * u + lane;
                if (v < vpt) x[u] = __ldcs(src + v);
            }
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const int v = base + 32 * u + lane;
                if (v >= vpt) continue;
                const int p = v / vpp;
                // first element of the vector in the destination [P][B][rows][Hl][128]
                const long e0 = ((long)((unsigned)p * a.B + b) * seq + n) * (vpp * 8) + (long)(v - p * vpp) * 8;
                if (!rot) {
                    __stcs(reinterpret_cast<uint4 *>(dst + e0 * 2), x[u]);
                    continue;
                }
                float f[8];
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&x[u]);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float2 e = __bfloat1622float2(h2[k]);
                    f[2 * k] = e.x * cs[k].x - e.y * cs[k].y;
                    f[2 * k + 1] = e.x * cs[k].y + e.y * cs[k].x;
                }
                if constexpr (std::is_same<TQK, __half>::value) {
#pragma unroll
                    for (int k = 0; k < 8; k++) bad |= !(fabsf(f[k]) < 65520.f);  // a finite half
                }
                if constexpr (sizeof(TQK) == 1) {
                    // e4m3, round to nearest even; beyond +-448 saturates and is reported
                    uint32_t w[2];
#pragma unroll
                    for (int k = 0; k < 8; k++) bad |= !(fabsf(f[k]) <= 448.f);
#pragma unroll
                    for (int k = 0; k < 2; k++) {
                        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k], f[4 * k + 1]), __NV_SATFINITE,
                                                                     __NV_E4M3);
                        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k + 2], f[4 * k + 3]),
                                                                     __NV_SATFINITE, __NV_E4M3);
                        w[k] = lo | (hi << 16);
                    }
                    __stcs(reinterpret_cast<uint2 *>(dst + e0), make_uint2(w[0], w[1]));
                } else {
                    uint4 y;
                    Vec<TQK>::store(&y, f);
                    __stcs(reinterpret_cast<uint4 *>(dst + e0 * 2), y);
                }
            }
        }
    }
    if (bad) atomicCAS(a.r.err, DEV_OK, DEV_RANGE);
}

// Rotary arguments of problem g: tensors q [B][S], k [B][Nv], joint_k [B][Nj]
// (rows of H*d), their destinations, tables and positions.
static RopeArgs rope_args(const Geom &g, const void *src_q, void *dst_q, const void *src_k, void *dst_k,
                          const void *src_jk, void *dst_jk, int *err) {
    RopeArgs a;
    a.err = err;
    a.src[0] = src_q, a.dst[0] = dst_q;
    a.src[1] = src_k, a.dst[1] = dst_k;
    a.src[2] = src_jk, a.dst[2] = dst_jk;
    a.tokens[0] = (long)g.B * g.S;
    a.tokens[1] = (long)g.B * g.Nv;
    a.tokens[2] = (long)g.B * g.Nj;
    a.seq[0] = g.S, a.seq[1] = g.Nv > 0 ? g.Nv : 1, a.seq[2] = g.Nj > 0 ? g.Nj : 1;
    a.Nv = g.Nv;
    a.H = g.H, a.d = g.d;
    a.grid_h = g.grid_h, a.grid_w = g.grid_w;
    a.seg1 = g.axis_dim[0] / 2;
    a.seg2 = (g.axis_dim[0] + g.axis_dim[1]) / 2;
    a.joint_rope = g.joint_rope;
    RopeLayout L = rope_layout(g);
    for (int t = 0; t < 4; t++) a.off[t] = L.off[t];
    for (int t = 0; t < 3; t++) a.half[t] = g.axis_dim[t] / 2;
    for (int t = 0; t < 3; t++) a.norm_w[t][0] = a.norm_w[t][1] = nullptr;
    a.eps = 0.f;
    return a;
}

cudaError_t launch_rope_split(const Geom &g, const float2 *tables, const void *const src[5], void *const dst[5],
                              int P, k6attn_dtype qk_out, int *err, cudaStream_t st) {
    SplitArgs a;
    a.r = rope_args(g, src[0], nullptr, src[1], nullptr, src[2], nullptr, err);
    const long cnt[5] = {(long)g.B * g.S, (long)g.B * g.Nv, (long)g.B * g.Nj, (long)g.B * g.Nv, (long)g.B * g.Nj};
    const long seq[5] = {g.S, g.Nv, g.Nj, g.Nv, g.Nj};
    long total = 0;
    for (int t = 0; t < 5; t++) {
        a.src[t] = src[t];
        a.dst[t] = dst[t];
        a.count[t] = cnt[t];
        a.seq[t] = seq[t] > 0 ? seq[t] : 1;
        total += cnt[t];
    }
    a.B = g.B, a.P = P, a.Hl = g.H / P;
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    auto launch = [&](auto kernel) {
        int per_sm = 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
        long blocks = (total + 7) / 8;  // one row per warp
        const long wave = (long)sms * (per_sm > 0 ? per_sm : 1);
        if (blocks > wave) blocks = wave;
        kernel<<<(unsigned)blocks, 256, 0, st>>>(a, tables);
    };
    if (qk_out == K6ATTN_F16) launch(rope_split_kernel<__half>);
    else if (qk_out == K6ATTN_E4M3) launch(rope_split_kernel<__nv_fp8_e4m3>);
    else launch(rope_split_kernel<__nv_bfloat16>);
    return cudaGetLastError();
}

cudaError_t launch_rope_qk(const Geom &g, const float2 *tables, const void *src_q, void *dst_q, const void *src_k,
                           void *dst_k, const void *src_jk, void *dst_jk, k6attn_dtype out_dtype, int *err,
                           cudaStream_t st, const QkNorm *norm) {
    RopeArgs a = rope_args(g, src_q, dst_q, src_k, dst_k, src_jk, dst_jk, err);
    const bool use_norm = norm != nullptr;
    a.eps = use_norm ? norm->eps : 0.f;
    for (int t = 0; t < 3; t++) a.norm_w[t][0] = a.norm_w[t][1] = nullptr;
    if (use_norm) {
        a.norm_w[0][0] = norm->q_w;
        a.norm_w[0][1] = norm->jq_w ? norm->jq_w : norm->q_w;
        a.norm_w[1][0] = a.norm_w[1][1] = norm->k_w;
        a.norm_w[2][0] = a.norm_w[2][1] = norm->jk_w ? norm->jk_w : norm->k_w;
    }
    long total = a.tokens[0] + a.tokens[1] + a.tokens[2];
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // one wave: as many 256-thread blocks as fit on the SMs at once (the kernel
    // strides over tokens), at most one token per warp
    auto launch = [&](auto kernel) {
        int per_sm = 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
        long blocks = (total + 7) / 8;
        const long wave = (long)sms * (per_sm > 0 ? per_sm : 1);
        if (blocks > wave) blocks = wave;
        kernel<<<(unsigned)blocks, 256, 0, st>>>(a, tables);
    };
    // short rows (fewer vectors than half of one warp pass): several rows per warp pass
    const int kpairs = g.dtype == K6ATTN_F32 ? 2 : 4;
    const int vpt = g.H * g.d / (2 * kpairs);
    if (!use_norm && 2 * vpt <= 32 * 6) {
        // lanes per row group, vectors per lane per row, rows per group pass (6 vectors in flight)
        const int vph = g.d / (2 * kpairs);
        const int gl = vph <= 16 ? 16 : 32;
        const int vpl = (vpt + gl - 1) / gl;
        const int rpg = 6 / vpl > 0 ? 6 / vpl : 1;
        const long rows_per_warp = (long)(32 / gl) * rpg;
        auto launch_short = [&](auto kernel) {
            int per_sm = 1;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
            long blocks = (total + 8L * rows_per_warp - 1) / (8L * rows_per_warp);
            const long wave = (long)sms * (per_sm > 0 ? per_sm : 1);
            if (blocks > wave) blocks = wave;
            kernel<<<(unsigned)blocks, 256, 0, st>>>(a, tables, gl, vpl, rpg);
        };
        if (g.dtype == K6ATTN_BF16 && out_dtype == K6ATTN_F16) launch_short(rope_short_kernel<__nv_bfloat16, __half>);
        else if (g.dtype == K6ATTN_BF16) launch_short(rope_short_kernel<__nv_bfloat16, __nv_bfloat16>);
        else launch_short(rope_short_kernel<float, float>);
        return cudaGetLastError();
    }
    if (g.dtype == K6ATTN_BF16 && out_dtype == K6ATTN_F16) {
        if (use_norm) launch(rope_kernel<__nv_bfloat16, __half, true>);
        else launch(rope_kernel<__nv_bfloat16, __half, false>);
    } else if (g.dtype == K6ATTN_BF16) {
        if (use_norm) launch(rope_kernel<__nv_bfloat16, __nv_bfloat16, true>);
        else launch(rope_kernel<__nv_bfloat16, __nv_bfloat16, false>);
    } else {
        if (use_norm) launch(rope_kernel<float, float, true>);
        else launch(rope_kernel<float, float, false>);
    }
    return cudaGetLastError();
}

}  // namespace k6
