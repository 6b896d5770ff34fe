// C-ABI layer: argument validation, the plan's device tables, and dispatch to
// the kernel launchers.  Declarations and contracts: include/cpdr.h.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <string>

#include "cpdr_internal.hpp"

namespace {

thread_local std::string g_last_error;

cpdr_status set_err(cpdr_status s, const std::string &msg) {
    g_last_error = msg;
    return s;
}

cpdr_status cuda_err(cudaError_t e, const char *what) {
    return set_err(CPDR_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                      cudaGetErrorString(e) + ")");
}

template <typename T>
cudaError_t upload(T **dst, const std::vector<T> &src) {
    *dst = nullptr;
    if (src.empty()) return cudaSuccess;
    cudaError_t e = cudaMalloc((void **)dst, sizeof(T) * src.size());
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src.data(), sizeof(T) * src.size(), cudaMemcpyHostToDevice);
}

void free_tables(cpdr::DeviceTables &t) {
    cudaFree(t.frags);
    cudaFree(t.pre_items);
    cudaFree(t.fwd_order);
    cudaFree(t.chains);
    cudaFree(t.zero_pre);
    cudaFree(t.zero_init);
    cudaFree(t.empty_seqs);
    cudaFree(t.frag_chunk0);
    cudaFree(t.wy_chunks);
    cudaFree(t.conv_tiles);
    cudaFree(t.host_items);
    cudaFree(t.bwd_pre_items);
    cudaFree(t.conv_halo);
    cudaFree(t.status);
    t = cpdr::DeviceTables();
}

void free_streams(cpdr_ctx *c) {
    for (void *&e : c->host_ev) {
        if (e) cudaEventDestroy((cudaEvent_t)e);
        e = nullptr;
    }
    if (c->copy_stream) cudaStreamDestroy((cudaStream_t)c->copy_stream);
    if (c->out_stream) cudaStreamDestroy((cudaStream_t)c->out_stream);
    c->copy_stream = c->out_stream = nullptr;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

cpdr_status check_ctx(const cpdr_ctx *c) {
    if (!c) return set_err(CPDR_ERR_INVALID, "null context");
    if (!c->has_device) return set_err(CPDR_ERR_INVALID, "context was created with CPDR_FLAG_HOST_ONLY");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    if (dev != c->device)
        return set_err(CPDR_ERR_INVALID, "current device differs from the device the context was created on");
    return CPDR_OK;
}

cpdr_status check_ptr(const void *p, const char *name, bool nullable = false) {
    if (!p) {
        if (nullable) return CPDR_OK;
        return set_err(CPDR_ERR_INVALID, std::string("null pointer: ") + name);
    }
    if (!aligned16(p)) return set_err(CPDR_ERR_INVALID, std::string("pointer not 16-byte aligned: ") + name);
    return CPDR_OK;
}

#define CPDR_TRY(x)                          \
    do {                                     \
        cpdr_status _s = (x);                \
        if (_s != CPDR_OK) return _s;        \
    } while (0)

cpdr_status launch_rc(int rc, const char *what) {
    if (rc != 0) return cuda_err((cudaError_t)rc, what);
    return CPDR_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct Sizes {
    size_t q, k, v, beta, gate, o, sext, m, sinit, fin;
};

Sizes sizes_of(const cpdr::Plan &p) {
    Sizes s;
    const size_t es = p.in_dtype == CPDR_DTYPE_F32 ? 4 : 2;
    const size_t tok = (size_t)p.B * (size_t)p.T;
    s.q = tok * p.Hq * p.dk * es;
    s.k = tok * p.H * p.dk * es;
    s.v = tok * p.H * p.dv * es;
    s.beta = tok * p.H * es;
    s.gate = tok * p.H * (p.gate_kind == CPDR_GATE_PER_DIM ? p.dk : 1) * sizeof(float);
    s.o = tok * p.Hq * p.dv * es;
    s.sext = (size_t)p.R * p.B * p.H * p.dk * p.dv * sizeof(float);
    s.m = (size_t)p.R * p.B * p.H * p.dk * p.dk * sizeof(float);
    s.sinit = s.sext;
    s.fin = (size_t)p.N * p.H * p.dk * p.dv * sizeof(float);
    return s;
}

}  // namespace

namespace cpdr {
// Records `msg` as this thread's last error and returns `s` (for other
// translation units of the library).
cpdr_status fail_with(cpdr_status s, const std::string &msg) { return set_err(s, msg); }
}  // namespace cpdr

extern "C" {

const char *cpdr_last_error(void) { return g_last_error.c_str(); }

const char *cpdr_version(void) { return "cpdr 0.1 (sm_103a)"; }

cpdr_status cpdr_ctx_create(const cpdr_desc *desc, cpdr_ctx **out) {
    if (!out) return set_err(CPDR_ERR_INVALID, "null output pointer");
    *out = nullptr;
    if (!desc) return set_err(CPDR_ERR_INVALID, "null descriptor");
    std::shared_ptr<cpdr::Plan> plan;
    try {
        plan = std::make_shared<cpdr::Plan>();
    } catch (const std::bad_alloc &) {
        return set_err(CPDR_ERR_INVALID, "out of host memory");
    }
    std::string err;
    cpdr_status s = cpdr::build_plan(*desc, *plan, err);
    if (s != CPDR_OK) return set_err(s, err);
    cpdr_ctx *c = new (std::nothrow) cpdr_ctx(std::move(plan));
    if (!c) return set_err(CPDR_ERR_INVALID, "out of host memory");
    c->use_tc = cpdr::tc_supported(c->plan) && !(desc->flags & CPDR_FLAG_FORCE_SIMT);
    if (!(desc->flags & CPDR_FLAG_HOST_ONLY)) {
        cudaError_t e = cudaGetDevice(&c->device);
        auto &p = c->plan;
        auto &t = c->dev;
        if (e == cudaSuccess) e = upload(&t.frags, p.frags);
        if (e == cudaSuccess) e = upload(&t.pre_items, p.pre_items);
        if (e == cudaSuccess) e = upload(&t.fwd_order, p.fwd_order);
        if (e == cudaSuccess) e = upload(&t.chains, p.chains);
        if (e == cudaSuccess) e = upload(&t.zero_pre, p.zero_pre);
        if (e == cudaSuccess) e = upload(&t.zero_init, p.zero_init);
        if (e == cudaSuccess) e = upload(&t.empty_seqs, p.empty_seqs);
        if (e == cudaSuccess) e = upload(&t.frag_chunk0, p.frag_chunk0);
        if (e == cudaSuccess) e = upload(&t.wy_chunks, p.wy_chunks);
        if (e == cudaSuccess) e = upload(&t.conv_tiles, p.conv_tiles);
        if (e == cudaSuccess) e = upload(&t.host_items, p.host_items);
        if (e == cudaSuccess) e = upload(&t.bwd_pre_items, p.bwd_pre_items);
        if (e == cudaSuccess) e = upload(&t.conv_halo, p.conv_halo);
        if (e == cudaSuccess) e = cudaMalloc((void **)&t.status, 64);
        if (e == cudaSuccess) e = cudaMemset(t.status, 0, 64);
        if (e == cudaSuccess) {
            cudaStream_t cs = nullptr, os = nullptr;
            e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
            c->copy_stream = cs;
            if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&os, cudaStreamNonBlocking);
            c->out_stream = os;
            for (int i = 0; i < cpdr_ctx::kHostEvents && e == cudaSuccess; i++) {
                cudaEvent_t ev = nullptr;
                e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
                c->host_ev[i] = ev;
            }
        }
        if (e != cudaSuccess) {
            free_tables(t);
            free_streams(c);
            delete c;
            return cuda_err(e, "cpdr_ctx_create: device tables");
        }
        c->has_device = true;
    }
    *out = c;
    return CPDR_OK;
}

void cpdr_ctx_destroy(cpdr_ctx *c) {
    if (!c) return;
    free_streams(c);
    if (c->has_device) free_tables(c->dev);
    delete c;
}

cpdr_status cpdr_buffer_sizes(const cpdr_ctx *c, size_t *sext, size_t *m, size_t *sinit, size_t *fin) {
    if (!c) return set_err(CPDR_ERR_INVALID, "null context");
    const Sizes s = sizes_of(c->plan);
    if (sext) *sext = s.sext;
    if (m) *m = s.m;
    if (sinit) *sinit = s.sinit;
    if (fin) *fin = s.fin;
    return CPDR_OK;
}

cpdr_status cpdr_plan_num_fragments(const cpdr_ctx *c, int32_t *n) {
    if (!c || !n) return set_err(CPDR_ERR_INVALID, "null argument");
    *n = (int32_t)c->plan.frags.size();
    return CPDR_OK;
}

cpdr_status cpdr_plan_fragments(const cpdr_ctx *c, cpdr_fragment *out, int32_t cap) {
    if (!c || (!out && cap > 0)) return set_err(CPDR_ERR_INVALID, "null argument");
    const int32_t n = (int32_t)c->plan.frags.size();
    for (int32_t i = 0; i < n && i < cap; i++) out[i] = c->plan.frags[i];
    return CPDR_OK;
}

cpdr_status cpdr_plan_counts(const cpdr_ctx *c, int32_t out[8]) {
    if (!c || !out) return set_err(CPDR_ERR_INVALID, "null argument");
    const auto &p = c->plan;
    out[0] = (int32_t)p.frags.size();
    out[1] = (int32_t)p.pre_items.size();
    out[2] = (int32_t)p.chains.size();
    out[3] = (int32_t)p.zero_pre.size();
    out[4] = (int32_t)p.zero_init.size();
    out[5] = (int32_t)p.empty_seqs.size();
    out[6] = cpdr::launches_per_step(c);
    out[7] = c->use_tc ? 1 : 0;
    return CPDR_OK;
}

cpdr_status cpdr_wy_bytes(const cpdr_ctx *c, size_t *bytes) {
    if (!c || !bytes) return set_err(CPDR_ERR_INVALID, "null argument");
    *bytes = cpdr::wy_bytes(c);
    return CPDR_OK;
}

cpdr_status cpdr_wy_build(const cpdr_ctx *c, const void *q, const void *k, const void *beta, const float *gate,
                          void *wy, void *stream) {
    CPDR_TRY(check_ctx(c));
    if (cpdr::wy_bytes(c) == 0) return CPDR_OK;
    const bool kda = c->plan.gate_kind == CPDR_GATE_PER_DIM;
    CPDR_TRY(check_ptr(q, "q", !kda));
    CPDR_TRY(check_ptr(k, "k"));
    CPDR_TRY(check_ptr(beta, "beta"));
    CPDR_TRY(check_ptr(gate, "gate"));
    CPDR_TRY(check_ptr(wy, "wy"));
    return launch_rc(kda ? cpdr::launch_tc_kda_prep(c, k, q, beta, gate, wy, stream)
                         : cpdr::launch_tc_wy(c, k, beta, gate, wy, stream),
                     "cpdr_wy_build");
}

cpdr_status cpdr_preprocess(const cpdr_ctx *c, const void *k, const void *v, const void *beta,
                            const float *gate, const void *wy, float *S_ext, float *M, void *stream) {
    CPDR_TRY(check_ctx(c));
    CPDR_TRY(check_ptr(k, "k"));
    CPDR_TRY(check_ptr(v, "v"));
    CPDR_TRY(check_ptr(beta, "beta"));
    CPDR_TRY(check_ptr(gate, "gate"));
    CPDR_TRY(check_ptr(wy, "wy", cpdr::wy_bytes(c) == 0));
    CPDR_TRY(check_ptr(S_ext, "S_ext"));
    CPDR_TRY(check_ptr(M, "M"));
    int rc = c->use_tc ? cpdr::launch_tc_pre(c, k, v, gate, wy, S_ext, M, stream)
                       : cpdr::launch_simt_pre(c, k, v, beta, gate, S_ext, M, stream);
    CPDR_TRY(launch_rc(rc, "cpdr_preprocess"));
    return launch_rc(cpdr::launch_zero_segments(c, S_ext, M, nullptr, nullptr, 0, stream),
                     "cpdr_preprocess: zero fill");
}

cpdr_status cpdr_merge(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init, void *stream) {
    CPDR_TRY(check_ctx(c));
    CPDR_TRY(check_ptr(S_ext, "S_ext"));
    CPDR_TRY(check_ptr(M, "M"));
    CPDR_TRY(check_ptr(S_init, "S_init"));
    CPDR_TRY(launch_rc(cpdr::launch_zero_segments(c, nullptr, nullptr, S_init, nullptr, 1, stream),
                       "cpdr_merge: zero fill"));
    return launch_rc(cpdr::launch_merge(c, S_ext, M, S_init, stream), "cpdr_merge");
}

cpdr_status cpdr_fwd(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta,
                     const float *gate, const void *wy, const float *S_init, void *o, float *final_state,
                     void *stream) {
    CPDR_TRY(check_ctx(c));
    CPDR_TRY(check_ptr(q, "q"));
    CPDR_TRY(check_ptr(k, "k"));
    CPDR_TRY(check_ptr(v, "v"));
    CPDR_TRY(check_ptr(beta, "beta"));
    CPDR_TRY(check_ptr(gate, "gate"));
    CPDR_TRY(check_ptr(wy, "wy", cpdr::wy_bytes(c) == 0));
    CPDR_TRY(check_ptr(S_init, "S_init"));
    CPDR_TRY(check_ptr(o, "o"));
    CPDR_TRY(check_ptr(final_state, "final_state", true));
    const int n = (int)c->plan.frags.size();
    int rc = c->use_tc ? cpdr::launch_tc_fwd(c, c->dev.fwd_order, n, q, k, v, gate, wy, S_init, o, final_state, stream)
                       : cpdr::launch_simt_fwd(c, c->dev.fwd_order, n, q, k, v, beta, gate, S_init, o, final_state,
                                               stream);
    CPDR_TRY(launch_rc(rc, "cpdr_fwd"));
    return launch_rc(cpdr::launch_zero_segments(c, nullptr, nullptr, nullptr, final_state, 2, stream),
                     "cpdr_fwd: zero fill");
}

cpdr_status cpdr_conv1d_fwd(const cpdr_ctx *c, const void *x, const float *weight, const float *bias,
                            int32_t channels, int32_t activation, void *y, void *stream) {
    CPDR_TRY(check_ctx(c));
    if (c->plan.conv_width < 1)
        return set_err(CPDR_ERR_INVALID, "cpdr_conv1d_fwd: the context was created without a conv width");
    if (channels < 1 || channels % 8 != 0)
        return set_err(CPDR_ERR_INVALID, "cpdr_conv1d_fwd: channels must be a positive multiple of 8");
    if (activation != 0 && activation != 1)
        return set_err(CPDR_ERR_INVALID, "cpdr_conv1d_fwd: activation must be 0 (none) or 1 (SiLU)");
    CPDR_TRY(check_ptr(x, "x"));
    CPDR_TRY(check_ptr(weight, "weight"));
    CPDR_TRY(check_ptr(bias, "bias", true));
    CPDR_TRY(check_ptr(y, "y"));
    const size_t es = c->plan.in_dtype == CPDR_DTYPE_F32 ? 4 : 2;
    const size_t nbytes = (size_t)c->plan.B * (size_t)c->plan.T * (size_t)channels * es;
    const char *xb = (const char *)x, *yb = (const char *)y;
    if (xb < yb + nbytes && yb < xb + nbytes) return set_err(CPDR_ERR_INVALID, "cpdr_conv1d_fwd: y overlaps x");
    return launch_rc(cpdr::launch_conv1d(c, x, weight, bias, channels, activation, y, stream), "cpdr_conv1d_fwd");
}

cpdr_status cpdr_bwd_workspace_bytes(const cpdr_ctx *c, size_t *bytes) {
    if (!c || !bytes) return set_err(CPDR_ERR_INVALID, "null argument");
    const Sizes s = sizes_of(c->plan);
    const size_t scratch = cpdr::bwd_uses_tc(c)
                               ? cpdr::bwd_tc_scratch_bytes(c)
                               : (size_t)cpdr::bwd_grid(c) * cpdr::bwd_scratch_floats_per_cta(c) * sizeof(float);
    *bytes = 2 * round256(s.sext) + round256(scratch);
    return CPDR_OK;
}

cpdr_status cpdr_bwd(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta,
                     const float *gate, const void *dout, const float *dht, const float *S_init, const float *M,
                     float *dq, float *dk, float *dv, float *dbeta, float *dgate, void *ws, size_t ws_bytes,
                     void *stream) {
    CPDR_TRY(check_ctx(c));
    const auto &p = c->plan;
    if (!cpdr::bwd_uses_tc(c) && !cpdr::bwd_simt_fits(c))
        return set_err(CPDR_ERR_UNSUPPORTED,
                       "cpdr_bwd: the query heads of one state do not fit the backward chain's shared memory");
    CPDR_TRY(check_ptr(q, "q"));
    CPDR_TRY(check_ptr(k, "k"));
    CPDR_TRY(check_ptr(v, "v"));
    CPDR_TRY(check_ptr(beta, "beta"));
    CPDR_TRY(check_ptr(gate, "gate"));
    CPDR_TRY(check_ptr(dout, "dout"));
    CPDR_TRY(check_ptr(dht, "dht", true));
    CPDR_TRY(check_ptr(S_init, "S_init"));
    CPDR_TRY(check_ptr(M, "M"));
    CPDR_TRY(check_ptr(dq, "dq"));
    CPDR_TRY(check_ptr(dk, "dk"));
    CPDR_TRY(check_ptr(dv, "dv"));
    CPDR_TRY(check_ptr(dbeta, "dbeta"));
    CPDR_TRY(check_ptr(dgate, "dgate"));
    CPDR_TRY(check_ptr(ws, "workspace"));
    size_t need = 0;
    cpdr_bwd_workspace_bytes(c, &need);
    if (ws_bytes < need) return set_err(CPDR_ERR_WORKSPACE, "cpdr_bwd: workspace too small");
    if (((uintptr_t)ws & 255u) != 0) return set_err(CPDR_ERR_INVALID, "cpdr_bwd: workspace not 256-byte aligned");
    const Sizes s = sizes_of(p);
    char *w = (char *)ws;
    float *dS_ext = (float *)w;
    float *dS_end = (float *)(w + round256(s.sext));
    float *scratch = (float *)(w + 2 * round256(s.sext));
    const size_t tok = (size_t)p.B * (size_t)p.T;
    cudaStream_t st = (cudaStream_t)stream;
    if (!cpdr::bwd_uses_tc(c)) {   // the CUDA-core chains add their sums atomically
        cudaError_t e = cudaMemsetAsync(dq, 0, tok * p.Hq * p.dk * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dk, 0, tok * p.H * p.dk * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, tok * p.H * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dgate, 0, s.gate, st);
        if (e != cudaSuccess) return cuda_err(e, "cpdr_bwd: zero fill");
    }
    return launch_rc(cpdr::launch_bwd(c, q, k, v, beta, gate, dout, dht, S_init, M, dS_ext, dS_end, scratch, dq, dk,
                                      dv, dbeta, dgate, stream),
                     "cpdr_bwd");
}

cpdr_status cpdr_plan_conv_tokens(const cpdr_ctx *c, int32_t *out, int32_t cap) {
    if (!c || (!out && cap > 0)) return set_err(CPDR_ERR_INVALID, "null argument");
    if (c->plan.conv_width < 1) return set_err(CPDR_ERR_INVALID, "the context was created without a conv width");
    const int32_t n = std::min<int32_t>(cap, (int32_t)c->plan.conv_pre_tokens.size());
    for (int32_t i = 0; i < n; i++) out[i] = c->plan.conv_pre_tokens[i];
    return CPDR_OK;
}

cpdr_status cpdr_host_workspace_bytes(const cpdr_ctx *c, size_t *bytes) {
    if (!c || !bytes) return set_err(CPDR_ERR_INVALID, "null argument");
    const Sizes s = sizes_of(c->plan);
    *bytes = round256(s.q) + round256(s.k) + round256(s.v) + round256(s.beta) + round256(s.gate) + round256(s.o) +
             round256(s.sext) + round256(s.m) + round256(s.sinit) + round256(s.fin) +
             round256(cpdr::wy_bytes(c));
    return CPDR_OK;
}

cpdr_status cpdr_forward_host(const cpdr_ctx *c, const void *q, const void *k, const void *v,
                              const void *beta, const float *gate, void *o, float *final_state,
                              void *ws, size_t ws_bytes, void *stream) {
    CPDR_TRY(check_ctx(c));
    if (!q || !k || !v || !beta || !gate || !o) return set_err(CPDR_ERR_INVALID, "null host pointer");
    CPDR_TRY(check_ptr(ws, "device_workspace"));
    size_t need = 0;
    cpdr_host_workspace_bytes(c, &need);
    if (ws_bytes < need) return set_err(CPDR_ERR_WORKSPACE, "device workspace too small");
    if (((uintptr_t)ws & 255u) != 0) return set_err(CPDR_ERR_INVALID, "device workspace not 256-byte aligned");
    const Sizes s = sizes_of(c->plan);
    char *p = (char *)ws;
    auto take = [&](size_t n) { char *r = p; p += round256(n); return r; };
    void *dq = take(s.q), *dk = take(s.k), *dv = take(s.v), *db = take(s.beta);
    float *dg = (float *)take(s.gate);
    void *dout = take(s.o);
    float *dse = (float *)take(s.sext), *dm = (float *)take(s.m), *dsi = (float *)take(s.sinit);
    float *dfin = (float *)take(s.fin);
    const size_t nwy = cpdr::wy_bytes(c);
    void *dwy = nwy ? take(nwy) : nullptr;
    cudaStream_t st = (cudaStream_t)stream, cs = (cudaStream_t)c->copy_stream, os = (cudaStream_t)c->out_stream;
    // A pipeline over three streams.  The inputs go over on the copy stream
    // in the order the stages need them -- k, beta, gate (the WY build; q
    // too for the per-dim gate), then v (the pre-process), then q group by
    // group -- and each stage on `stream` waits only for its own inputs: the
    // WY build, pre-process and merge run while v and q are in transit, the
    // forward runs group by group (kHostParts groups of consecutive tokens)
    // as q arrives, and each group's o goes back on the output stream while
    // the next group runs.  The copy stream starts after everything enqueued
    // on `stream` before the call; `stream` ends after the last copy back.
    const auto &pl = c->plan;
    const bool kda = pl.gate_kind == CPDR_GATE_PER_DIM;
    auto ev = [&](int i) { return (cudaEvent_t)c->host_ev[i]; };
    constexpr int E_START = 0, E_IN0 = 1, E_IN1 = 2, E_OUT = 3, E_Q = 4, E_F = 4 + cpdr::kHostParts;
    const size_t q_tok = s.q / ((size_t)pl.B * (size_t)pl.T), o_tok = s.o / ((size_t)pl.B * (size_t)pl.T);
    cudaError_t e = cudaEventRecord(ev(E_START), st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev(E_START), 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, k, s.k, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaMemcpyAsync(db, beta, s.beta, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dg, gate, s.gate, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess && kda) e = cudaMemcpyAsync(dq, q, s.q, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(ev(E_IN0), cs);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, v, s.v, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(ev(E_IN1), cs);
    for (int g = 0; g < cpdr::kHostParts && e == cudaSuccess; g++) {
        const size_t t0 = (size_t)pl.host_part_tok[g], t1 = (size_t)pl.host_part_tok[g + 1];
        if (!kda && t1 > t0)
            e = cudaMemcpyAsync((char *)dq + t0 * q_tok, (const char *)q + t0 * q_tok, (t1 - t0) * q_tok,
                                cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(ev(E_Q + g), cs);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev(E_IN0), 0);
    if (e != cudaSuccess) return cuda_err(e, "cpdr_forward_host: host-to-device copy");
    CPDR_TRY(cpdr_wy_build(c, dq, dk, db, dg, dwy, stream));
    e = cudaStreamWaitEvent(st, ev(E_IN1), 0);
    if (e != cudaSuccess) return cuda_err(e, "cpdr_forward_host: stream wait");
    CPDR_TRY(cpdr_preprocess(c, dk, dv, db, dg, dwy, dse, dm, stream));
    CPDR_TRY(cpdr_merge(c, dse, dm, dsi, stream));
    for (int g = 0; g < cpdr::kHostParts; g++) {
        const int off = pl.host_part_off[g], n = pl.host_part_off[g + 1] - off;
        const size_t t0 = (size_t)pl.host_part_tok[g], t1 = (size_t)pl.host_part_tok[g + 1];
        e = cudaStreamWaitEvent(st, ev(E_Q + g), 0);
        if (e != cudaSuccess) return cuda_err(e, "cpdr_forward_host: stream wait");
        const int32_t *items = c->dev.host_items + off;
        int rc = c->use_tc ? cpdr::launch_tc_fwd(c, items, n, dq, dk, dv, dg, dwy, dsi, dout, dfin, stream)
                           : cpdr::launch_simt_fwd(c, items, n, dq, dk, dv, db, dg, dsi, dout, dfin, stream);
        CPDR_TRY(launch_rc(rc, "cpdr_forward_host: forward"));
        e = cudaEventRecord(ev(E_F + g), st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(os, ev(E_F + g), 0);
        if (e == cudaSuccess && t1 > t0)
            e = cudaMemcpyAsync((char *)o + t0 * o_tok, (const char *)dout + t0 * o_tok, (t1 - t0) * o_tok,
                                cudaMemcpyDeviceToHost, os);
        if (e != cudaSuccess) return cuda_err(e, "cpdr_forward_host: device-to-host copy");
    }
    CPDR_TRY(launch_rc(cpdr::launch_zero_segments(c, nullptr, nullptr, nullptr, dfin, 2, stream),
                       "cpdr_forward_host: zero fill"));
    if (final_state) {
        e = cudaMemcpyAsync(final_state, dfin, s.fin, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_err(e, "cpdr_forward_host: device-to-host copy");
    }
    e = cudaEventRecord(ev(E_OUT), os);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev(E_OUT), 0);
    if (e != cudaSuccess) return cuda_err(e, "cpdr_forward_host: stream wait");
    return CPDR_OK;
}

cpdr_status cpdr_check_device_status(const cpdr_ctx *c, void *stream) {
    if (!c) return set_err(CPDR_ERR_INVALID, "null context");
    int32_t *word = nullptr;
    if (c->has_device) {
        CPDR_TRY(check_ctx(c));
        word = c->dev.status;
    } else {
        // a host-only context has no status word of its own: its kernels ran
        // through the allocation-free entry point, whose array holds the word
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
        word = cpdr::noalloc_status_word(dev);
        if (!word) return CPDR_OK;   // nothing has run on this device
    }
    int32_t h[16];
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(h, word, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_err(e, "cpdr_check_device_status");
    if (h[0] != 0) {
        cudaMemsetAsync(word, 0, 64, st);
        cudaStreamSynchronize(st);
        char buf[160];
        snprintf(buf, sizeof(buf), "a bounded device wait gave up: code %d (site %d, block %d)", h[0], h[1], h[2]);
        return set_err(CPDR_ERR_TIMEOUT, buf);
    }
    return CPDR_OK;
}

}  // extern "C"
