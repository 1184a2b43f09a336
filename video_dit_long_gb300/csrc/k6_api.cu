// k6_api.cu -- the C ABI of libk6attn: handle, argument checks, workspace
// layout and the launch sequence of one forward pass.  Every check runs on
// the host before any launch; nothing here aborts.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "k6attn.h"
#include "k6_internal.h"

struct k6attn_handle {
    k6attn_desc desc;
    k6::Geom g;
    float2 *tables = nullptr;
    size_t table_bytes = 0;
    int *err = nullptr;                 // device error word
    unsigned long long wait_limit_ns = 2000000000ull;
    int strict_order = 0;
    int rotate_bf16 = 0;                // forward: rotated copies in bf16 instead of fp16
    int device = 0;
};

namespace k6 {

static thread_local char g_msg[512];

k6attn_status set_error(k6attn_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

k6attn_status cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return K6ATTN_OK;
    return set_error(K6ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

struct WsLayout {
    size_t q_rot = 0, k_rot = 0, jk_rot = 0, part_o = 0, part_lse = 0, total = 0;
};

static WsLayout ws_layout(const Geom &g, int n, bool rope) {
    WsLayout L;
    size_t off = 0;
    const size_t row = (size_t)g.H * g.d;
    if (rope) {
        L.q_rot = off;
        off += round256((size_t)g.B * g.S * row * g.elem);
        L.k_rot = off;
        off += round256((size_t)g.B * g.Nv * row * g.elem);
        L.jk_rot = off;
        off += round256((size_t)g.B * g.Nj * row * g.elem);
    }
    if (n > 1) {
        L.part_o = off;
        off += round256((size_t)n * g.B * g.Sq * row * 4);
        L.part_lse = off;
        off += round256((size_t)n * g.B * g.H * g.Sq * 4);
    }
    L.total = off;
    return L;
}

// The attention kernels on rotated inputs: n_chunks == 1 writes out/lse,
// n_chunks > 1 writes fp32 partials into out/lse (see k6attn_attention_chunks).
// With group > 0 and merge, each CTA's `group` consecutive chunks leave one
// partial (n_chunks / group partials; the output itself when that is 1).
static k6attn_status run_attention(k6attn_handle *h, const Geom &g, const void *q, const void *k, const void *v,
                                   const void *jk, const void *jv, bool qk_f16, int n_chunks, void *out, float *lse,
                                   cudaStream_t st, const float *row_bound = nullptr, int group = 0,
                                   bool merge = false, bool qk8 = false) {
    if (g.elem == 2) {
        AttnTcOptions opt{h->wait_limit_ns, h->err,    h->strict_order, qk_f16 ? 1 : 0, row_bound,
                          qk8 ? 1 : 0,      group,     merge ? 1 : 0};
        const char *why = nullptr;
        // the single-tile kernel (one 128-row Q tile per CTA), for bf16, fp16 and e4m3 q/k
        cudaError_t e = launch_attn_tc_single(g, q, k, v, jk, jv, n_chunks, out, lse, opt, st, &why);
        if (e != cudaSuccess) {
            if (why) return set_error(K6ATTN_ERR_CUDA, "attention: %s", why);
            return cuda_check(e, "attention launch");
        }
        return K6ATTN_OK;
    }
    const size_t o_stride = (size_t)g.B * g.Sq * g.H * g.d, l_stride = (size_t)g.B * g.H * g.Sq;
    return cuda_check(launch_attn_f32(g, static_cast<const float *>(q), static_cast<const float *>(k),
                                      static_cast<const float *>(v), static_cast<const float *>(jk),
                                      static_cast<const float *>(jv), n_chunks, static_cast<float *>(out), o_stride,
                                      lse, l_stride, st),
                      "fp32 attention launch");
}

// Chunks per CTA, and so partials per chunk count, for problem g: bf16 handles
// merge each CTA's chunk group in the kernel; the fp32 kernel writes one
// partial per chunk.
static int group_for(const Geom &g, int n_chunks) { return g.elem == 2 ? chunk_group(g, n_chunks) : 1; }

// Attention over n_chunks K/V chunks, then the log-sum-exp merge of what is
// left: n_chunks / group partials (k6attn_forward, k6attn_cross_forward).
// part_o / part_lse are workspace regions sized for n_chunks partials.
static k6attn_status attention_and_merge(k6attn_handle *h, const Geom &g, const void *q, const void *k, const void *v,
                                         const void *jk, const void *jv, bool qk_f16, int n_chunks, void *out,
                                         float *lse, char *part_o, char *part_lse, cudaStream_t st, const char *fn) {
    const int group = group_for(g, n_chunks);
    const int parts = n_chunks / group;
    if (parts == 1) return run_attention(h, g, q, k, v, jk, jv, qk_f16, n_chunks, out, lse, st, nullptr, group, true);
    float *po = reinterpret_cast<float *>(part_o), *pl = reinterpret_cast<float *>(part_lse);
    k6attn_status s = run_attention(h, g, q, k, v, jk, jv, qk_f16, n_chunks, po, pl, st, nullptr, group, true);
    if (s != K6ATTN_OK) return s;
    const cudaError_t e = launch_lse_merge(g, parts, po, pl, out, lse, st);
    if (e != cudaSuccess) return set_error(K6ATTN_ERR_CUDA, "%s: merge launch: %s", fn, cudaGetErrorString(e));
    return K6ATTN_OK;
}

// Checks shared by the two attention entry points.
static k6attn_status check_inputs(const char *fn, const Geom &g, const void *q, const void *k, const void *v,
                                  const void *jk, const void *jv, int n_chunks, const void *out, size_t out_bytes,
                                  const float *lse, size_t lse_bytes, int qk_elem = 0) {
    if (!q || !k || !v || !out) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: null q, k, v or out", fn);
    if (g.Nj > 0 && (!jk || !jv))
        return set_error(K6ATTN_ERR_INVALID_ARG, "%s: %ld joint tokens but joint_k/joint_v is null", fn, g.Nj);
    if (n_chunks < 1) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: n_chunks must be >= 1", fn);
    if (g.S % n_chunks)
        return set_error(K6ATTN_ERR_INVALID_ARG, "%s: sequence length %ld is not divisible by %d chunks", fn, g.S,
                         n_chunks);
    const void *ptrs[] = {q, k, v, jk, jv, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
    if (reinterpret_cast<uintptr_t>(lse) & 3) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: lse misaligned", fn);
    const size_t row = (size_t)g.H * g.d * g.elem;
    const size_t qkrow = (size_t)g.H * g.d * (qk_elem ? qk_elem : g.elem);  // q/k/joint_k may be narrower
    const size_t qb = g.B * g.Sq * qkrow, kb = g.B * g.Nv * qkrow, jkb = g.B * g.Nj * qkrow;
    const size_t vb = g.B * g.Nv * row, jvb = g.B * g.Nj * row;
    const void *ins[] = {q, k, v, jk, jv};
    const size_t insz[] = {qb, kb, vb, jkb, jvb};
    for (int i = 0; i < 5; i++)
        if (overlap(out, out_bytes, ins[i], insz[i]) || overlap(lse, lse_bytes, ins[i], insz[i]))
            return set_error(K6ATTN_ERR_INVALID_ARG, "%s: out or lse overlaps an input", fn);
    if (overlap(out, out_bytes, lse, lse_bytes)) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: out overlaps lse", fn);
    return K6ATTN_OK;
}

// The q/k type an attention call may take with this handle: the handle's own,
// and F16 or E4M3 for BF16 handles.  Bytes per q/k element, or 0 (refused,
// message set).
static int qk_bytes(const char *fn, const Geom &g, k6attn_dtype qk) {
    if (qk == g.dtype) return g.elem;
    if (g.dtype == K6ATTN_BF16 && qk == K6ATTN_F16) return 2;
    if (g.dtype == K6ATTN_BF16 && qk == K6ATTN_E4M3) return 1;
    set_error(K6ATTN_ERR_INVALID_ARG, "%s: q/k type %d not allowed for this handle", fn, (int)qk);
    return 0;
}

k6attn_status check_handle(const char *fn, k6attn_t h) {
    if (!h) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: null handle", fn);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return set_error(K6ATTN_ERR_CUDA, "%s: no current device", fn);
    if (dev != h->device)
        return set_error(K6ATTN_ERR_INVALID_ARG, "%s: the handle was created on device %d but device %d is current",
                         fn, h->device, dev);
    return K6ATTN_OK;
}

}  // namespace k6

using namespace k6;

extern "C" {

const char *k6attn_status_string(k6attn_status s) {
    switch (s) {
        case K6ATTN_OK: return "ok";
        case K6ATTN_ERR_INVALID_ARG: return "invalid argument";
        case K6ATTN_ERR_UNSUPPORTED: return "unsupported";
        case K6ATTN_ERR_CUDA: return "CUDA error";
        case K6ATTN_ERR_TIMEOUT: return "device wait timed out";
        case K6ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case K6ATTN_ERR_RANGE: return "rotated value out of fp16 range";
    }
    return "unknown status";
}

const char *k6attn_last_error(void) { return g_msg; }

k6attn_status k6attn_create(const k6attn_desc *desc, k6attn_t *out) {
    g_msg[0] = 0;
    if (!desc || !out) return set_error(K6ATTN_ERR_INVALID_ARG, "create: null descriptor or output pointer");
    *out = nullptr;
    const k6attn_desc &d = *desc;
    if (d.B < 1 || d.H < 1 || d.grid_t < 1 || d.grid_h < 1 || d.grid_w < 1 || d.n_joint < 0)
        return set_error(K6ATTN_ERR_INVALID_ARG, "create: B, H and the grid must be >= 1, n_joint >= 0");
    if (d.dtype != K6ATTN_BF16 && d.dtype != K6ATTN_F32)
        return set_error(K6ATTN_ERR_INVALID_ARG, "create: unknown dtype %d", (int)d.dtype);
    if (d.d != 64 && d.d != 128) return set_error(K6ATTN_ERR_UNSUPPORTED, "create: head dim %d (want 64 or 128)", d.d);
    if (d.dtype == K6ATTN_BF16 && d.d != 128)
        return set_error(K6ATTN_ERR_UNSUPPORTED, "create: bf16 path needs head dim 128 (got %d)", d.d);
    int sum = 0;
    for (int a = 0; a < 3; a++) {
        if (d.axis_dim[a] < 0 || (d.axis_dim[a] & 1))
            return set_error(K6ATTN_ERR_INVALID_ARG, "create: axis_dim[%d] = %d must be even and >= 0", a,
                             d.axis_dim[a]);
        sum += d.axis_dim[a];
    }
    if (sum != d.d) return set_error(K6ATTN_ERR_INVALID_ARG, "create: axis dims sum to %d, head dim is %d", sum, d.d);
    if (!(d.theta > 0.0)) return set_error(K6ATTN_ERR_INVALID_ARG, "create: theta must be > 0");
    if (d.joint_rope != 0 && d.joint_rope != 1)
        return set_error(K6ATTN_ERR_INVALID_ARG, "create: joint_rope must be 0 or 1");
    const long Nv = (long)d.grid_t * d.grid_h * d.grid_w;
    const long S = Nv + d.n_joint;
    // TMA coordinates and several index products are 32-bit
    if (S >= (1L << 30) || (long)d.B * S * d.H >= (1L << 31))
        return set_error(K6ATTN_ERR_UNSUPPORTED, "create: problem too large (B*S*H = %ld)", (long)d.B * S * d.H);

    k6attn_handle *h = new k6attn_handle();
    h->desc = d;
    Geom &g = h->g;
    g.B = d.B, g.H = d.H, g.d = d.d;
    g.Nv = Nv, g.Nj = d.n_joint, g.S = S, g.Sq = S;
    g.grid_t = d.grid_t, g.grid_h = d.grid_h, g.grid_w = d.grid_w;
    for (int a = 0; a < 3; a++) g.axis_dim[a] = d.axis_dim[a];
    g.joint_rope = d.joint_rope;
    g.elem = d.dtype == K6ATTN_BF16 ? 2 : 4;
    g.dtype = d.dtype;
    cudaGetDevice(&h->device);
    RopeLayout L = rope_layout(g);
    h->table_bytes = (size_t)L.total * sizeof(float2);
    k6attn_status st = cuda_check(cudaMalloc(&h->err, sizeof(int)), "create: error word");
    if (st == K6ATTN_OK) st = cuda_check(cudaMemset(h->err, 0, sizeof(int)), "create: error word");
    if (st == K6ATTN_OK && h->table_bytes)
        st = cuda_check(cudaMalloc(&h->tables, h->table_bytes), "create: rotary tables");
    if (st == K6ATTN_OK) st = cuda_check(launch_rope_tables(g, d.theta, h->tables, 0), "create: rotary tables");
    if (st == K6ATTN_OK) st = cuda_check(cudaDeviceSynchronize(), "create: rotary tables");
    if (st != K6ATTN_OK) {
        cudaFree(h->tables);
        cudaFree(h->err);
        delete h;
        return st;
    }
    *out = h;
    return K6ATTN_OK;
}

void k6attn_destroy(k6attn_t h) {
    if (!h) return;
    // free on the handle's own device, whichever device the caller has current
    int cur = -1;
    const bool other = cudaGetDevice(&cur) == cudaSuccess && cur != h->device;
    if (other) cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->tables);
    cudaFree(h->err);
    if (other) cudaSetDevice(cur);
    delete h;
}

const void *k6attn_rope_tables(k6attn_t h) { return h ? h->tables : nullptr; }
size_t k6attn_rope_tables_bytes(k6attn_t h) { return h ? h->table_bytes : 0; }

size_t k6attn_workspace_bytes(k6attn_t h, int n_chunks, int with_rope) {
    if (!h || n_chunks < 1) return 0;
    return ws_layout(h->g, n_chunks, with_rope != 0).total;
}

k6attn_status k6attn_set_option(k6attn_t h, k6attn_option opt, long long value) {
    if (!h) return set_error(K6ATTN_ERR_INVALID_ARG, "set_option: null handle");  // host-side only
    if (value < 0) return set_error(K6ATTN_ERR_INVALID_ARG, "set_option: negative value");
    switch (opt) {
        case K6ATTN_OPT_WAIT_LIMIT_NS: h->wait_limit_ns = (unsigned long long)value; return K6ATTN_OK;
        case K6ATTN_OPT_STRICT_MMA_ORDER: h->strict_order = value ? 1 : 0; return K6ATTN_OK;
        case K6ATTN_OPT_ROTATE_BF16: h->rotate_bf16 = value ? 1 : 0; return K6ATTN_OK;
    }
    return set_error(K6ATTN_ERR_INVALID_ARG, "set_option: unknown option %d", (int)opt);
}

// Shared checks and launch of the two rotary entry points.
static k6attn_status rope_common(const char *fn, k6attn_t h, const void *q, const void *k, const void *joint_k,
                                 const void *rope_tables, void *q_out, void *k_out, void *joint_k_out,
                                 k6attn_dtype out_dtype, const QkNorm *norm, void *stream) {
    {
        k6attn_status hs = check_handle(fn, h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (!q || !k || !q_out || !k_out || (g.Nj > 0 && (!joint_k || !joint_k_out)) || (!rope_tables && h->table_bytes))
        return set_error(K6ATTN_ERR_INVALID_ARG, "%s: null tensor or table pointer", fn);
    if (out_dtype != g.dtype && !(g.dtype == K6ATTN_BF16 && out_dtype == K6ATTN_F16))
        return set_error(K6ATTN_ERR_INVALID_ARG, "%s: output type %d not allowed for this handle", fn, (int)out_dtype);
    const void *ptrs[] = {q, k, joint_k, q_out, k_out, joint_k_out, rope_tables};
    for (const void *p : ptrs)
        if (!aligned16(p)) return set_error(K6ATTN_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
    const size_t row = (size_t)g.H * g.d * g.elem;
    const size_t nb[3] = {g.B * g.S * row, g.B * g.Nv * row, g.B * g.Nj * row};
    const void *src[3] = {q, k, joint_k};
    const void *dst[3] = {q_out, k_out, joint_k_out};
    for (int a = 0; a < 3; a++) {
        if (dst[a] == src[a] && nb[a] && out_dtype != g.dtype)
            return set_error(K6ATTN_ERR_INVALID_ARG, "%s: in-place rotation keeps the handle's type", fn);
        for (int b = 0; b < 3; b++) {
            if (a != b && (overlap(src[a], nb[a], src[b], nb[b]) || overlap(dst[a], nb[a], dst[b], nb[b])))
                return set_error(K6ATTN_ERR_INVALID_ARG, "%s: tensors overlap", fn);
            if (dst[a] != src[a] && overlap(dst[a], nb[a], src[b], nb[b]))
                return set_error(K6ATTN_ERR_INVALID_ARG, "%s: an output overlaps an input", fn);
        }
    }
    return cuda_check(launch_rope_qk(g, static_cast<const float2 *>(rope_tables), q, q_out, k, k_out, joint_k,
                                     joint_k_out, out_dtype, h->err, static_cast<cudaStream_t>(stream), norm),
                      "rope launch");
}

k6attn_status k6attn_rope_qk(k6attn_t h, const void *q, const void *k, const void *joint_k, const void *rope_tables,
                             void *q_out, void *k_out, void *joint_k_out, k6attn_dtype out_dtype, void *stream) {
    g_msg[0] = 0;
    return rope_common("rope_qk", h, q, k, joint_k, rope_tables, q_out, k_out, joint_k_out, out_dtype, nullptr,
                       stream);
}

k6attn_status k6attn_norm_rope_qk(k6attn_t h, const void *q, const void *k, const void *joint_k,
                                  const float *q_weight, const float *k_weight, const float *joint_q_weight,
                                  const float *joint_k_weight, float eps, const void *rope_tables, void *q_out,
                                  void *k_out, void *joint_k_out, k6attn_dtype out_dtype, void *stream) {
    g_msg[0] = 0;
    if (!q_weight || !k_weight) return set_error(K6ATTN_ERR_INVALID_ARG, "norm_rope_qk: null q or k weight");
    if (!(eps >= 0.f)) return set_error(K6ATTN_ERR_INVALID_ARG, "norm_rope_qk: eps must be >= 0");
    const uintptr_t al = reinterpret_cast<uintptr_t>(q_weight) | reinterpret_cast<uintptr_t>(k_weight) |
                         reinterpret_cast<uintptr_t>(joint_q_weight) | reinterpret_cast<uintptr_t>(joint_k_weight);
    if (al & 3) return set_error(K6ATTN_ERR_INVALID_ARG, "norm_rope_qk: weights must be 4-byte aligned");
    QkNorm norm{q_weight, joint_q_weight, k_weight, joint_k_weight, eps};
    return rope_common("norm_rope_qk", h, q, k, joint_k, rope_tables, q_out, k_out, joint_k_out, out_dtype, &norm,
                       stream);
}

size_t k6attn_row_bounds_bytes(k6attn_t h) {
    if (!h) return 0;
    return ((size_t)h->g.B * h->g.H * h->g.Sq + (size_t)h->g.B * h->g.H) * sizeof(float);
}

k6attn_status k6attn_row_bounds(k6attn_t h, const void *q, const void *k, const void *joint_k, k6attn_dtype qk_dtype,
                                float *bounds, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("row_bounds", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (!q || !k || !bounds || (g.Nj > 0 && !joint_k))
        return set_error(K6ATTN_ERR_INVALID_ARG, "row_bounds: null pointer");
    if (qk_dtype != g.dtype && !(g.dtype == K6ATTN_BF16 && qk_dtype == K6ATTN_F16))
        return set_error(K6ATTN_ERR_INVALID_ARG, "row_bounds: q/k type %d not allowed for this handle", (int)qk_dtype);
    if (!aligned16(q) || !aligned16(k) || !aligned16(joint_k) || (reinterpret_cast<uintptr_t>(bounds) & 3))
        return set_error(K6ATTN_ERR_INVALID_ARG, "row_bounds: misaligned pointer");
    const size_t row = (size_t)g.H * g.d * (qk_dtype == K6ATTN_F32 ? 4 : 2);
    const size_t bb = k6attn_row_bounds_bytes(h);
    if (overlap(bounds, bb, q, g.B * g.Sq * row) || overlap(bounds, bb, k, g.B * g.Nv * row) ||
        overlap(bounds, bb, joint_k, g.B * g.Nj * row))
        return set_error(K6ATTN_ERR_INVALID_ARG, "row_bounds: bounds overlap an input");
    return cuda_check(launch_row_bounds(g, qk_dtype, q, k, joint_k, bounds, static_cast<cudaStream_t>(stream)),
                      "row_bounds launch");
}

k6attn_status k6attn_attention_chunks_bounded(k6attn_t h, const void *q, const void *k, const void *v,
                                              const void *joint_k, const void *joint_v, k6attn_dtype qk_dtype,
                                              const float *bounds, int n_chunks, void *out, float *lse,
                                              void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("attention_chunks_bounded", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (g.dtype != K6ATTN_BF16)
        return set_error(K6ATTN_ERR_UNSUPPORTED, "attention_chunks_bounded: the constant-max path is bf16 only");
    if (!bounds || (reinterpret_cast<uintptr_t>(bounds) & 3))
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunks_bounded: null or misaligned bounds");
    if (n_chunks > 1 && !lse)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunks_bounded: partial lse is required when n_chunks > 1");
    if (qk_dtype != K6ATTN_BF16 && qk_dtype != K6ATTN_F16)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunks_bounded: q/k type %d", (int)qk_dtype);
    const int n = n_chunks > 1 ? n_chunks : 1;
    const size_t ob = (size_t)n * g.B * g.Sq * g.H * g.d * (n_chunks > 1 ? 4 : g.elem);
    const size_t lb = (size_t)n * g.B * g.H * g.Sq * 4;
    k6attn_status s = check_inputs("attention_chunks_bounded", g, q, k, v, joint_k, joint_v, n_chunks, out, ob, lse, lb);
    if (s != K6ATTN_OK) return s;
    const size_t bb = k6attn_row_bounds_bytes(h);
    if (overlap(bounds, bb, out, ob) || overlap(bounds, bb, lse, lb))
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunks_bounded: bounds overlap an output");
    return run_attention(h, g, q, k, v, joint_k, joint_v, qk_dtype == K6ATTN_F16, n_chunks, out, lse,
                         static_cast<cudaStream_t>(stream), bounds);
}

k6attn_status k6attn_attention_chunk_groups_bounded(k6attn_t h, const void *q, const void *k, const void *v,
                                                    const void *joint_k, const void *joint_v, k6attn_dtype qk_dtype,
                                                    const float *bounds, int n_chunks, int group, void *out,
                                                    float *lse, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("attention_chunk_groups_bounded", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (g.dtype != K6ATTN_BF16)
        return set_error(K6ATTN_ERR_UNSUPPORTED, "attention_chunk_groups_bounded: the constant-max path is bf16 only");
    if (!bounds || (reinterpret_cast<uintptr_t>(bounds) & 3))
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunk_groups_bounded: null or misaligned bounds");
    if (group < 1 || n_chunks < 1 || n_chunks % group)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunk_groups_bounded: group %d must divide n_chunks %d",
                         group, n_chunks);
    const int parts = n_chunks / group;
    if (parts > 1 && !lse)
        return set_error(K6ATTN_ERR_INVALID_ARG,
                         "attention_chunk_groups_bounded: partial lse is required when n_chunks / group > 1");
    if (qk_dtype != K6ATTN_BF16 && qk_dtype != K6ATTN_F16)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunk_groups_bounded: q/k type %d", (int)qk_dtype);
    const size_t ob = (size_t)parts * g.B * g.Sq * g.H * g.d * (parts > 1 ? 4 : g.elem);
    const size_t lb = (size_t)parts * g.B * g.H * g.Sq * 4;
    k6attn_status s =
        check_inputs("attention_chunk_groups_bounded", g, q, k, v, joint_k, joint_v, n_chunks, out, ob, lse, lb);
    if (s != K6ATTN_OK) return s;
    const size_t bb = k6attn_row_bounds_bytes(h);
    if (overlap(bounds, bb, out, ob) || overlap(bounds, bb, lse, lb))
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunk_groups_bounded: bounds overlap an output");
    return run_attention(h, g, q, k, v, joint_k, joint_v, qk_dtype == K6ATTN_F16, n_chunks, out, lse,
                         static_cast<cudaStream_t>(stream), bounds, group, true);
}

k6attn_status k6attn_lse_merge(k6attn_t h, const float *part_o, const float *part_lse, int n_chunks, void *out,
                               float *lse, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("lse_merge", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (!part_o || !part_lse || !out) return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge: null pointer");
    if (n_chunks < 1) return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge: n_chunks must be >= 1");
    if (!aligned16(part_o) || !aligned16(out) || (reinterpret_cast<uintptr_t>(part_lse) & 3) ||
        (reinterpret_cast<uintptr_t>(lse) & 3))
        return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge: partials/out must be 16-byte aligned, lse 4-byte");
    const size_t po = (size_t)n_chunks * g.B * g.S * g.H * g.d * 4, pl = (size_t)n_chunks * g.B * g.H * g.S * 4;
    const size_t ob = (size_t)g.B * g.S * g.H * g.d * g.elem, lb = (size_t)g.B * g.H * g.S * 4;
    if (overlap(out, ob, part_o, po) || overlap(out, ob, part_lse, pl) || overlap(lse, lb, part_o, po) ||
        overlap(lse, lb, part_lse, pl) || overlap(out, ob, lse, lb))
        return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge: outputs overlap the partials");
    return cuda_check(launch_lse_merge(g, n_chunks, part_o, part_lse, out, lse, static_cast<cudaStream_t>(stream)),
                      "lse_merge launch");
}

k6attn_status k6attn_forward(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                             const void *joint_v, const void *rope_tables, int n_chunks, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("forward", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qb = (size_t)g.B * g.S * g.H * g.d * g.elem, lb = (size_t)g.B * g.H * g.S * 4;
    k6attn_status s = check_inputs("forward", g, q, k, v, joint_k, joint_v, n_chunks, out, qb, lse, lb);
    if (s != K6ATTN_OK) return s;
    if (!aligned16(rope_tables) || !aligned16(workspace))
        return set_error(K6ATTN_ERR_INVALID_ARG, "forward: pointers must be 16-byte aligned");
    const bool rope = rope_tables != nullptr;
    const WsLayout L = ws_layout(g, n_chunks, rope);
    if (L.total) {
        if (!workspace || workspace_bytes < L.total)
            return set_error(K6ATTN_ERR_WORKSPACE, "forward: workspace of %zu bytes needed, %zu given", L.total,
                             workspace ? workspace_bytes : (size_t)0);
        const size_t row = (size_t)g.H * g.d * g.elem;
        const void *ins[] = {q, k, v, joint_k, joint_v};
        const size_t insz[] = {g.B * g.S * row, g.B * g.Nv * row, g.B * g.Nv * row, g.B * g.Nj * row,
                               g.B * g.Nj * row};
        for (int i = 0; i < 5; i++)
            if (overlap(workspace, L.total, ins[i], insz[i]))
                return set_error(K6ATTN_ERR_INVALID_ARG, "forward: workspace overlaps an input");
        if (overlap(workspace, L.total, out, qb) || overlap(workspace, L.total, lse, lb))
            return set_error(K6ATTN_ERR_INVALID_ARG, "forward: workspace overlaps out or lse");
    }
    char *ws = static_cast<char *>(workspace);
    const void *qa = q, *ka = k, *jka = joint_k;
    if (rope) {
        void *qr = ws + L.q_rot, *kr = ws + L.k_rot, *jkr = g.Nj ? ws + L.jk_rot : nullptr;
        // a bf16 handle keeps its rotated copies in fp16 (8x finer rounding of the logits' inputs)
        // unless asked to keep bf16's range
        s = cuda_check(launch_rope_qk(g, static_cast<const float2 *>(rope_tables), q, qr, k, kr, joint_k, jkr,
                                      g.dtype == K6ATTN_BF16 && !h->rotate_bf16 ? K6ATTN_F16 : g.dtype, h->err, st),
                       "forward: rope launch");
        if (s != K6ATTN_OK) return s;
        qa = qr, ka = kr, jka = jkr;
    }
    const bool qk_f16 = rope && g.dtype == K6ATTN_BF16 && !h->rotate_bf16;
    return attention_and_merge(h, g, qa, ka, v, jka, joint_v, qk_f16, n_chunks, out, lse, ws + L.part_o,
                               ws + L.part_lse, st, "forward");
}

k6attn_status k6attn_attention_chunks(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                                      const void *joint_v, k6attn_dtype qk_dtype, int n_chunks, void *out, float *lse,
                                      void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("attention_chunks", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (n_chunks > 1 && !lse)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunks: partial lse is required when n_chunks > 1");
    const int n = n_chunks > 1 ? n_chunks : 1;
    const size_t ob = (size_t)n * g.B * g.S * g.H * g.d * (n_chunks > 1 ? 4 : g.elem);
    const size_t lb = (size_t)n * g.B * g.H * g.S * 4;
    const int qkb = qk_bytes("attention_chunks", g, qk_dtype);
    if (!qkb) return K6ATTN_ERR_INVALID_ARG;
    k6attn_status s = check_inputs("attention_chunks", g, q, k, v, joint_k, joint_v, n_chunks, out, ob, lse, lb, qkb);
    if (s != K6ATTN_OK) return s;
    return run_attention(h, g, q, k, v, joint_k, joint_v, qk_dtype == K6ATTN_F16, n_chunks, out, lse,
                         static_cast<cudaStream_t>(stream), nullptr, 0, false, qk_dtype == K6ATTN_E4M3);
}

int k6attn_chunk_group(k6attn_t h, int n_chunks) {
    if (!h || n_chunks < 1) return 0;
    return group_for(h->g, n_chunks);
}

k6attn_status k6attn_attention_chunk_groups(k6attn_t h, const void *q, const void *k, const void *v,
                                            const void *joint_k, const void *joint_v, k6attn_dtype qk_dtype,
                                            int n_chunks, int group, void *out, float *lse, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("attention_chunk_groups", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (group < 1 || n_chunks < 1 || n_chunks % group)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunk_groups: group %d must divide n_chunks %d", group,
                         n_chunks);
    if (group > 1 && g.elem != 2)
        return set_error(K6ATTN_ERR_UNSUPPORTED, "attention_chunk_groups: chunk groups need a bf16 handle");
    const int parts = n_chunks / group;
    if (parts > 1 && !lse)
        return set_error(K6ATTN_ERR_INVALID_ARG, "attention_chunk_groups: partial lse is required when "
                                                 "n_chunks / group > 1");
    const int qkb = qk_bytes("attention_chunk_groups", g, qk_dtype);
    if (!qkb) return K6ATTN_ERR_INVALID_ARG;
    const size_t ob = (size_t)parts * g.B * g.S * g.H * g.d * (parts > 1 ? 4 : g.elem);
    const size_t lb = (size_t)parts * g.B * g.H * g.S * 4;
    k6attn_status s =
        check_inputs("attention_chunk_groups", g, q, k, v, joint_k, joint_v, n_chunks, out, ob, lse, lb, qkb);
    if (s != K6ATTN_OK) return s;
    return run_attention(h, g, q, k, v, joint_k, joint_v, qk_dtype == K6ATTN_F16, n_chunks, out, lse,
                         static_cast<cudaStream_t>(stream), nullptr, group, true, qk_dtype == K6ATTN_E4M3);
}

k6attn_status k6attn_rope_split_heads(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                                      const void *joint_v, const void *rope_tables, int P, k6attn_dtype qk_out_dtype,
                                      void *q_out, void *k_out, void *v_out, void *joint_k_out, void *joint_v_out,
                                      void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("rope_split_heads", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (g.dtype != K6ATTN_BF16)
        return set_error(K6ATTN_ERR_UNSUPPORTED, "rope_split_heads: needs a bf16 handle (d = 128)");
    if (qk_out_dtype != K6ATTN_BF16 && qk_out_dtype != K6ATTN_F16 && qk_out_dtype != K6ATTN_E4M3)
        return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: rotated q/k type must be BF16, F16 or E4M3");
    if (P < 1 || g.H % P)
        return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: %d heads are not divisible by %d", g.H, P);
    if (!q || !k || !v || !q_out || !k_out || !v_out || (!rope_tables && h->table_bytes))
        return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: null tensor or table pointer");
    if (g.Nj > 0 && (!joint_k || !joint_v || !joint_k_out || !joint_v_out))
        return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: %ld joint tokens but a joint pointer is null",
                         g.Nj);
    const void *src[5] = {q, k, joint_k, v, joint_v};
    void *dst[5] = {q_out, k_out, joint_k_out, v_out, joint_v_out};
    const size_t row = (size_t)g.H * g.d * 2, orow = (size_t)g.H * g.d * (qk_out_dtype == K6ATTN_E4M3 ? 1 : 2);
    const size_t nb[5] = {g.B * g.S * row, g.B * g.Nv * row, g.B * g.Nj * row, g.B * g.Nv * row, g.B * g.Nj * row};
    const size_t ob[5] = {g.B * g.S * orow, g.B * g.Nv * orow, g.B * g.Nj * orow, g.B * g.Nv * row,
                          g.B * g.Nj * row};
    for (int a = 0; a < 5; a++) {
        if (!aligned16(src[a]) || !aligned16(dst[a]))
            return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: pointers must be 16-byte aligned");
        for (int b = 0; b < 5; b++) {
            if (overlap(dst[a], ob[a], src[b], nb[b]))
                return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: an output overlaps an input");
            if (a != b && overlap(dst[a], ob[a], dst[b], ob[b]))
                return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: outputs overlap");
        }
    }
    if (!aligned16(rope_tables))
        return set_error(K6ATTN_ERR_INVALID_ARG, "rope_split_heads: rotary tables must be 16-byte aligned");
    return cuda_check(launch_rope_split(g, static_cast<const float2 *>(rope_tables), src, dst, P, qk_out_dtype, h->err,
                                        static_cast<cudaStream_t>(stream)),
                      "rope_split_heads launch");
}

k6attn_status k6attn_lse_merge_heads(k6attn_t h, const float *part_o, const float *part_lse, int n_parts, int P,
                                     void *out, float *lse, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("lse_merge_heads", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (!part_o || !part_lse || !out) return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge_heads: null pointer");
    if (n_parts < 1) return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge_heads: n_parts must be >= 1");
    if (P < 1 || g.H % P)
        return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge_heads: %d heads are not divisible by %d", g.H, P);
    if (!aligned16(part_o) || !aligned16(out) || (reinterpret_cast<uintptr_t>(part_lse) & 3) ||
        (reinterpret_cast<uintptr_t>(lse) & 3))
        return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge_heads: partials/out must be 16-byte aligned, lse 4-byte");
    const size_t po = (size_t)n_parts * g.B * g.S * g.H * g.d * 4, pl = (size_t)n_parts * g.B * g.H * g.S * 4;
    const size_t ob = (size_t)g.B * g.S * g.H * g.d * g.elem, lb = (size_t)g.B * g.H * g.S * 4;
    if (overlap(out, ob, part_o, po) || overlap(out, ob, part_lse, pl) || overlap(lse, lb, part_o, po) ||
        overlap(lse, lb, part_lse, pl) || overlap(out, ob, lse, lb))
        return set_error(K6ATTN_ERR_INVALID_ARG, "lse_merge_heads: outputs overlap the partials");
    return cuda_check(launch_lse_merge(g, n_parts, part_o, part_lse, out, lse, static_cast<cudaStream_t>(stream), P),
                      "lse_merge_heads launch");
}

size_t k6attn_backward_workspace_bytes(k6attn_t h) {
    if (!h) return 0;
    return (((size_t)h->g.B * h->g.H * h->g.S * sizeof(float2)) + 255) & ~(size_t)255;
}

k6attn_status k6attn_backward(k6attn_t h, const void *q, const void *k, const void *v, const void *joint_k,
                              const void *joint_v, k6attn_dtype qk_dtype, const void *out, const void *dout,
                              const float *lse, float *dq, float *dk, float *dv, float *djoint_k, float *djoint_v,
                              void *workspace, size_t workspace_bytes, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("backward", h);
        if (hs != K6ATTN_OK) return hs;
    }
    const Geom &g = h->g;
    if (g.dtype != K6ATTN_BF16 || g.d != 128)
        return set_error(K6ATTN_ERR_UNSUPPORTED, "backward: needs a BF16 handle with d = 128");
    if (qk_dtype != K6ATTN_BF16 && qk_dtype != K6ATTN_F16)
        return set_error(K6ATTN_ERR_INVALID_ARG, "backward: q/k type must be BF16 or F16");
    if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv)
        return set_error(K6ATTN_ERR_INVALID_ARG, "backward: null pointer");
    if (g.Nj > 0 && (!joint_k || !joint_v || !djoint_k || !djoint_v))
        return set_error(K6ATTN_ERR_INVALID_ARG, "backward: %ld joint tokens but a joint pointer is null", g.Nj);
    const void *ptrs[] = {q, k, v, joint_k, joint_v, out, dout, dq, dk, dv, djoint_k, djoint_v, workspace};
    for (const void *p : ptrs)
        if (!aligned16(p)) return set_error(K6ATTN_ERR_INVALID_ARG, "backward: pointers must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(lse) & 3) return set_error(K6ATTN_ERR_INVALID_ARG, "backward: lse misaligned");
    const size_t need = k6attn_backward_workspace_bytes(h);
    if (!workspace || workspace_bytes < need)
        return set_error(K6ATTN_ERR_WORKSPACE, "backward: workspace of %zu bytes needed, %zu given", need,
                         workspace ? workspace_bytes : (size_t)0);
    const size_t row16 = (size_t)g.H * g.d * 2, row32 = (size_t)g.H * g.d * 4;
    const size_t qb = g.B * g.S * row16, kvb = g.B * g.Nv * row16, jb = g.B * g.Nj * row16;
    const void *ins[] = {q, k, v, joint_k, joint_v, out, dout, lse};
    const size_t insz[] = {qb, kvb, kvb, jb, jb, qb, qb, (size_t)g.B * g.H * g.S * 4};
    const void *outs[] = {dq, dk, dv, djoint_k, djoint_v, workspace};
    const size_t outsz[] = {g.B * g.S * row32, g.B * g.Nv * row32, g.B * g.Nv * row32, g.B * g.Nj * row32,
                            g.B * g.Nj * row32, need};
    for (int i = 0; i < 6; i++) {
        for (int j = 0; j < 8; j++)
            if (overlap(outs[i], outsz[i], ins[j], insz[j]))
                return set_error(K6ATTN_ERR_INVALID_ARG, "backward: an output overlaps an input");
        for (int j = i + 1; j < 6; j++)
            if (overlap(outs[i], outsz[i], outs[j], outsz[j]))
                return set_error(K6ATTN_ERR_INVALID_ARG, "backward: two outputs overlap");
    }
    const char *why = nullptr;
    cudaError_t e = launch_attn_bwd(g, qk_dtype == K6ATTN_F16, q, k, v, joint_k, joint_v, out, dout, lse,
                                    static_cast<float2 *>(workspace), dq, dk, dv, djoint_k, djoint_v,
                                    h->wait_limit_ns, h->err, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) {
        if (why) return set_error(K6ATTN_ERR_CUDA, "backward: %s", why);
        return cuda_check(e, "backward launch");
    }
    return K6ATTN_OK;
}

// Cross-attention from at most one 128-row query tile (the single-tile kernel)
// reads every K/V byte once for a few query rows, so it is bound by HBM, and
// the B*H*n CTAs of n chunks can leave the last wave nearly empty (24 heads x 8
// chunks = 192 CTAs on 152 SMs: the second wave streams through 40 SMs).  The
// chunks are then split into m sub-chunks each (merged like chunks: the result
// is the same attention), m <= 4 chosen to waste the least of the last wave
// while every sub-chunk keeps at least 1024 keys.
constexpr int CROSS_SPLIT_MAX = 4;
static int cross_split(const Geom &g, int n_chunks) {
    if (g.Sq > 128 || g.elem != 2) return 1;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long units = (long)g.B * g.H * n_chunks;
    int best = 1;
    double best_waves = (double)((units + sms - 1) / sms);  // waves of full-chunk CTAs
    for (int m = 2; m <= CROSS_SPLIT_MAX; m++) {
        if (g.S % ((long)n_chunks * m) || g.S / ((long)n_chunks * m) < 1024) continue;
        const double waves = (double)((units * m + sms - 1) / sms) / m;
        if (waves < best_waves - 1e-9) best = m, best_waves = waves;
    }
    return best;
}

// The handle's batch, heads, head dim and type with Sq query rows over Sk keys.
static Geom cross_geom(const Geom &base, long Sq, long Sk) {
    Geom g = base;
    g.Nv = Sk, g.Nj = 0, g.S = Sk, g.Sq = Sq;
    g.grid_t = 1, g.grid_h = 1, g.grid_w = (int)(Sk < (1L << 30) ? Sk : 1);
    g.joint_rope = 0;
    return g;
}

size_t k6attn_cross_workspace_bytes(k6attn_t h, long Sq, int n_chunks) {
    if (!h || n_chunks < 1 || Sq < 1) return 0;
    // a short query range may be split into up to CROSS_SPLIT_MAX sub-chunks per chunk
    const int most = Sq <= 128 && h->g.elem == 2 ? n_chunks * CROSS_SPLIT_MAX : n_chunks;
    return ws_layout(cross_geom(h->g, Sq, 1), most, false).total;
}

k6attn_status k6attn_cross_forward(k6attn_t h, const void *q, long Sq, const void *k, const void *v, long Sk,
                                   int n_chunks, void *out, float *lse, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("cross_forward", h);
        if (hs != K6ATTN_OK) return hs;
    }
    if (Sq < 1 || Sk < 1) return set_error(K6ATTN_ERR_INVALID_ARG, "cross_forward: Sq and Sk must be >= 1");
    if (Sq >= (1L << 30) || Sk >= (1L << 30) || (long)h->g.B * Sq * h->g.H >= (1L << 31) ||
        (long)h->g.B * Sk * h->g.H >= (1L << 31))
        return set_error(K6ATTN_ERR_UNSUPPORTED, "cross_forward: problem too large");
    const Geom g = cross_geom(h->g, Sq, Sk);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qb = (size_t)g.B * Sq * g.H * g.d * g.elem, lb = (size_t)g.B * g.H * Sq * 4;
    k6attn_status s = check_inputs("cross_forward", g, q, k, v, nullptr, nullptr, n_chunks, out, qb, lse, lb);
    if (s != K6ATTN_OK) return s;
    if (!aligned16(workspace)) return set_error(K6ATTN_ERR_INVALID_ARG, "cross_forward: workspace misaligned");
    // chunks as the kernels run them; the finer split only where the caller's workspace holds it
    int m = cross_split(g, n_chunks);
    if (m > 1 && (!workspace || workspace_bytes < ws_layout(g, n_chunks * m, false).total)) m = 1;
    const int n_int = n_chunks * m;
    if (n_int == 1) return run_attention(h, g, q, k, v, nullptr, nullptr, false, 1, out, lse, st);
    const WsLayout L = ws_layout(g, n_int, false);
    if (!workspace || workspace_bytes < L.total)
        return set_error(K6ATTN_ERR_WORKSPACE, "cross_forward: workspace of %zu bytes needed, %zu given", L.total,
                         workspace ? workspace_bytes : (size_t)0);
    const size_t kvb = (size_t)g.B * Sk * g.H * g.d * g.elem;
    if (overlap(workspace, L.total, q, qb) || overlap(workspace, L.total, k, kvb) ||
        overlap(workspace, L.total, v, kvb) || overlap(workspace, L.total, out, qb) ||
        overlap(workspace, L.total, lse, lb))
        return set_error(K6ATTN_ERR_INVALID_ARG, "cross_forward: workspace overlaps a tensor");
    char *ws = static_cast<char *>(workspace);
    return attention_and_merge(h, g, q, k, v, nullptr, nullptr, false, n_int, out, lse, ws + L.part_o,
                               ws + L.part_lse, st, "cross_forward");
}

k6attn_status k6attn_seq2head_relayout(const void *src, void *dst, int B, long S, int H, int d, int elem_bytes,
                                       int P, int direction, void *stream) {
    g_msg[0] = 0;
    if (!src || !dst) return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: null pointer");
    if (B < 1 || S < 1 || H < 1 || d < 1 || P < 1)
        return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: B, S, H, d, P must be >= 1");
    if (elem_bytes != 2 && elem_bytes != 4) return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: elem_bytes 2 or 4");
    if (direction != 0 && direction != 1) return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: direction 0 or 1");
    if (S % P)
        return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: sequence length %ld is not divisible by %d", S, P);
    if (H % P) return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: %d heads are not divisible by %d", H, P);
    if ((long long)P * B * S >= (1LL << 31) || (long long)(H / P) * d * elem_bytes >= (1LL << 31))
        return set_error(K6ATTN_ERR_UNSUPPORTED, "relayout: too large");
    if (!aligned16(src) || !aligned16(dst))
        return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: pointers must be 16-byte aligned");
    const size_t bytes = (size_t)B * S * H * d * elem_bytes;
    if (overlap(src, bytes, dst, bytes)) return set_error(K6ATTN_ERR_INVALID_ARG, "relayout: src and dst overlap");
    return cuda_check(launch_relayout(src, dst, B, S, H, d, elem_bytes, P, direction, static_cast<cudaStream_t>(stream)),
                      "relayout launch");
}

k6attn_status k6attn_sync(k6attn_t h, void *stream) {
    g_msg[0] = 0;
    {
        k6attn_status hs = check_handle("sync", h);
        if (hs != K6ATTN_OK) return hs;
    }
    k6attn_status s = cuda_check(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "sync");
    if (s != K6ATTN_OK) return s;
    int word = 0;
    s = cuda_check(cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost), "sync: error word");
    if (s != K6ATTN_OK) return s;
    if (word) {
        cudaMemset(h->err, 0, sizeof(int));
        if (word == DEV_RANGE) return set_error(K6ATTN_ERR_RANGE, "a rotated q/k value does not fit fp16");
        if (word == DEV_LAYOUT)
            return set_error(K6ATTN_ERR_CUDA, "the device placed the attention kernel's shared memory off a 1024-byte boundary");
        return set_error(K6ATTN_ERR_TIMEOUT, "a device-side wait gave up (code %d)", word);
    }
    return K6ATTN_OK;
}

}  // extern "C"
