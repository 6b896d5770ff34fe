// Allocation-free whole-path entry point (cpdr_forward_noalloc).
//
// Some callers cannot allocate device memory at all: for example code that
// runs inside a runtime which owns every byte of device memory through its
// own pool or static memory plan, where an allocation would break the plan,
// or a process that must keep its device footprint fixed after start-up.
// Such callers cannot create the caller-owned exchange buffers (S_ext, M,
// S_init) nor let the context allocate its device tables.  This entry point
// serves them: it keeps everything the path needs besides the caller's
// inputs and outputs -- the status word of the bounded waits, the plan
// tables, the WY tiles and the three exchange buffers -- in one file-scope device array
// of fixed size, and calls no allocating routine.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "cpdr_internal.hpp"

namespace {

// Fixed maximum of the static scratch: 32 MiB per device.  Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_cpdr_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;                 // serialises the set-up and the use of the array
void *g_scratch_addr[256] = {};  // device address of the array, per device (set up once)

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" cpdr_status cpdr_forward_noalloc(const cpdr_ctx *c, const void *q, const void *k, const void *v,
                                            const void *beta, const float *gate, void *o, float *final_state,
                                            void *stream) {
    if (!c) return cpdr::fail_with(CPDR_ERR_INVALID, "null context");
    if (!q || !k || !v || !beta || !gate || !o) return cpdr::fail_with(CPDR_ERR_INVALID, "null device pointer");
    const cpdr::Plan &p = c->plan;
    // scratch layout: status word | plan tables | S_ext | M | S_init | WY tiles
    const size_t n_frag = p.frags.size(), n_pre = p.pre_items.size(), n_ch = p.chains.size();
    const size_t b_status = 256;
    const size_t b_frags = round256(n_frag * sizeof(cpdr_fragment));
    const size_t b_pre = round256(n_pre * sizeof(int32_t)), b_ord = round256(n_frag * sizeof(int32_t));
    const size_t b_ch = round256(n_ch * sizeof(cpdr::MergeChain));
    const size_t b_zp = round256(p.zero_pre.size() * sizeof(int32_t));
    const size_t b_zi = round256(p.zero_init.size() * sizeof(int32_t));
    const size_t b_es = round256(p.empty_seqs.size() * sizeof(int32_t));
    const size_t b_c0 = round256(p.frag_chunk0.size() * sizeof(int32_t));
    const size_t b_wc = round256(p.wy_chunks.size() * sizeof(cpdr::WyChunk));
    const size_t b_wy = round256(cpdr::wy_bytes(c));
    const size_t per_seg = (size_t)p.R * p.B * p.H * p.dk;
    const size_t b_sext = round256(per_seg * p.dv * sizeof(float)), b_m = round256(per_seg * p.dk * sizeof(float));
    const size_t need =
        b_status + b_frags + b_pre + b_ord + b_ch + b_zp + b_zi + b_es + b_c0 + b_wc + 2 * b_sext + b_m + b_wy;
    if (need > kNoAllocScratchBytes) {
        char buf[256];
        snprintf(buf, sizeof(buf),
                 "cpdr_forward_noalloc: this problem needs %zu bytes of device scratch (exchange buffers "
                 "R*B*H*dk*(2*dv+dk)*4 bytes, WY tiles and plan tables); the allocation-free entry point holds at "
                 "most %zu",
                 need, kNoAllocScratchBytes);
        return cpdr::fail_with(CPDR_ERR_WORKSPACE, buf);
    }
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 256)
        return cpdr::fail_with(CPDR_ERR_CUDA, "cpdr_forward_noalloc: no current device");
    if (!g_scratch_addr[dev]) {
        // set-up, once per device, with that device current: the array's
        // host-side name is not a device address; ask the runtime for it
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_cpdr_noalloc_scratch);
        if (e != cudaSuccess || !addr)
            return cpdr::fail_with(CPDR_ERR_CUDA, std::string("cpdr_forward_noalloc: cudaGetSymbolAddress: ") +
                                                      cudaGetErrorString(e));
        g_scratch_addr[dev] = addr;
    }
    char *base = static_cast<char *>(g_scratch_addr[dev]);
    cpdr::DeviceTables t;
    char *cur = base;
    auto take = [&](size_t n) { char *r = cur; cur += n; return r; };
    int32_t *array_status = reinterpret_cast<int32_t *>(take(b_status));
    t.frags = reinterpret_cast<cpdr_fragment *>(take(b_frags));
    t.pre_items = reinterpret_cast<int32_t *>(take(b_pre));
    t.fwd_order = reinterpret_cast<int32_t *>(take(b_ord));
    t.chains = reinterpret_cast<cpdr::MergeChain *>(take(b_ch));
    t.zero_pre = reinterpret_cast<int32_t *>(take(b_zp));
    t.zero_init = reinterpret_cast<int32_t *>(take(b_zi));
    t.empty_seqs = reinterpret_cast<int32_t *>(take(b_es));
    t.frag_chunk0 = reinterpret_cast<int32_t *>(take(b_c0));
    t.wy_chunks = reinterpret_cast<cpdr::WyChunk *>(take(b_wc));
    float *S_ext = reinterpret_cast<float *>(take(b_sext));
    float *M = reinterpret_cast<float *>(take(b_m));
    float *S_init = reinterpret_cast<float *>(take(b_sext));
    void *wy = b_wy ? take(b_wy) : nullptr;
    // Expired waits go to the context's own status word when it has one (a
    // regular context), else to the array's; cpdr_check_device_status reads
    // whichever of the two the context has.  The array keeps the previous
    // call's contents: clear its status word, copy this context's tables
    // (the exchange buffers are fully written by the stages).
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaSuccess;
    if (c->has_device) {
        if (dev != c->device)
            return cpdr::fail_with(CPDR_ERR_INVALID,
                                   "cpdr_forward_noalloc: current device differs from the context's device");
        t.status = c->dev.status;
    } else {
        t.status = array_status;
        e = cudaMemsetAsync(array_status, 0, b_status, st);
    }
    auto put = [&](void *dst, const void *src, size_t n) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st);
    };
    put(t.frags, p.frags.data(), n_frag * sizeof(cpdr_fragment));
    put(t.pre_items, p.pre_items.data(), n_pre * sizeof(int32_t));
    put(t.fwd_order, p.fwd_order.data(), n_frag * sizeof(int32_t));
    put(t.chains, p.chains.data(), n_ch * sizeof(cpdr::MergeChain));
    put(t.zero_pre, p.zero_pre.data(), p.zero_pre.size() * sizeof(int32_t));
    put(t.zero_init, p.zero_init.data(), p.zero_init.size() * sizeof(int32_t));
    put(t.empty_seqs, p.empty_seqs.data(), p.empty_seqs.size() * sizeof(int32_t));
    put(t.frag_chunk0, p.frag_chunk0.data(), p.frag_chunk0.size() * sizeof(int32_t));
    put(t.wy_chunks, p.wy_chunks.data(), p.wy_chunks.size() * sizeof(cpdr::WyChunk));
    if (e != cudaSuccess)
        return cpdr::fail_with(CPDR_ERR_CUDA, std::string("cpdr_forward_noalloc: table upload: ") + cudaGetErrorString(e));
    // Run the three stages on a view of the context that points at the
    // array's tables: the view shares the caller's plan and leaves the
    // caller's context untouched.  Every stage runs on the caller's stream
    // (the view has no copy streams of its own).
    cpdr_ctx view(*c);
    view.dev = t;
    view.has_device = true;
    view.device = dev;
    view.copy_stream = view.out_stream = nullptr;
    for (void *&ev : view.host_ev) ev = nullptr;
    cpdr_status s = cpdr_wy_build(&view, q, k, beta, gate, wy, stream);
    if (s == CPDR_OK) s = cpdr_preprocess(&view, k, v, beta, gate, wy, S_ext, M, stream);
    if (s == CPDR_OK) s = cpdr_merge(&view, S_ext, M, S_init, stream);
    if (s == CPDR_OK) s = cpdr_fwd(&view, q, k, v, beta, gate, wy, S_init, o, final_state, stream);
    return s;
}

namespace cpdr {
// Status word of the array on device `dev` (nullptr until the allocation-free
// entry point has been set up there).
int32_t *noalloc_status_word(int dev) {
    if (dev < 0 || dev >= 256) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    return static_cast<int32_t *>(g_scratch_addr[dev]);
}
}  // namespace cpdr
