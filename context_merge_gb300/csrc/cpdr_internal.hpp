// Internal declarations shared by the C-ABI layer, the host planner and the
// kernel launchers.  Nothing here is visible through include/cpdr.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <memory>
#include <string>
#include <vector>

#include "../../include/cpdr.h"

namespace cpdr {

constexpr int kChunk = 64;      // chunk size fixed by the article's Code Flow (chunk_size=64)
constexpr int kHostParts = 4;   // token groups of the host-buffer path's pipeline

// A chain of segments r0 < r1 of one row b crossed by one sequence: the merge
// scan writes S_init for segments r0+1 .. r1 ([FLA-CP] §2.1 merge, §5.2).
struct MergeChain {
    int32_t b, r0, r1, pad;
};

// One chunk of one fragment (the unit of the WY build): first token on the
// flattened axis and its number of valid rows (<= 64; the rest is padding).
struct WyChunk {
    int64_t tok0;
    int32_t nv, pad;
};

// Causal-conv1d work unit: up to kConvTile tokens of one fragment (memory
// positions tok0 .. tok0 + n - 1).  halo says where the conv_width - 1 inputs
// before tok0 come from: kHaloMemory = the tokens right before tok0 (same
// fragment), kHaloZero = none (the sequence starts at tok0), k >= 0 = row k
// of the halo table (memory positions, -1 for positions before the sequence).
constexpr int kConvTile = 64;
constexpr int kMaxConvWidth = 8;
constexpr int32_t kHaloMemory = -2, kHaloZero = -1;
struct ConvTile {
    int64_t tok0;
    int32_t n, halo;
};

// Bytes of the WY tiles of one (chunk, head): T' = T diag(beta), and
// T'' = T diag(beta gamma) as a bf16 hi/lo pair, each a 64 x 64 bf16 tile
// stored as the 128-byte-swizzled shared-memory image the MMA reads.
constexpr size_t kWyTileBytes = 8192;
constexpr size_t kWyUnitBytes = 3 * kWyTileBytes;

// Per-dim gate (KDA) units: the WY tiles (with gamma = 1: the gate lives in
// the operand tiles), then the per-dim decay 2^(G_C) and the gated operand
// tiles of the chunk, each 64 rows x 128 columns bf16 as two 8 KiB swizzled
// 64-column images: Kg = k 2^G (hi, lo), Kgam = k 2^(G_C - G) (hi, lo),
// Qg = q 2^G, and the masked intra-chunk product P = (Q K^T ⊙ Lambda)
// (64 x 64, one image).  Offsets are multiples of 1 KiB (swizzle atoms).
constexpr size_t kKdaOffGC = 3 * kWyTileBytes;          // 128 fp32 (1 KiB slot)
constexpr size_t kKdaOffKg = kKdaOffGC + 1024;
constexpr size_t kKdaOffKgam = kKdaOffKg + 16384;
constexpr size_t kKdaOffKgLo = kKdaOffKgam + 16384;
constexpr size_t kKdaOffKgamLo = kKdaOffKgLo + 16384;
constexpr size_t kKdaOffQg = kKdaOffKgamLo + 16384;
constexpr size_t kKdaOffP = kKdaOffQg + 16384;
constexpr size_t kKdaUnitBytes = kKdaOffP + kWyTileBytes;   // 113 KiB
static_assert(kKdaUnitBytes % 1024 == 0, "KDA unit must keep 1 KiB alignment");
// Grouped query heads (G query heads per state head): the unit holds Qg and
// P of its state's first query head; those of query heads 1 .. G-1 follow
// all units, laid out as in the unit, [chunk][head][G - 1] x 24 KiB.
constexpr size_t kKdaQpBytes = kKdaUnitBytes - kKdaOffQg;

// Host plan ([FLA-CP] §3.2-§3.3): fragments per segment and the derived
// work lists.  All token indices are on the flattened [B*T] axis.
struct Plan {
    int32_t B = 0, H = 0, dk = 0, dv = 0, N = 0;
    int32_t Hq = 0, G = 1;   // query heads of q and o, and query heads per state (Hq = G H)
    bool vfirst = false;     // dk x dv state buffers stored [dv, dk]
    int32_t R = 0;           // segments per row: the ranks, or 2 x ranks (zigzag pieces)
    int64_t T = 0;           // tokens per row (or packed total)
    int64_t L = 0;           // segment length
    int32_t gate_kind = 0, in_dtype = 0;
    uint32_t flags = 0;
    float scale = 1.f;
    bool packed = false;
    std::vector<int64_t> cu;                 // N+1 offsets on the flattened axis
    std::vector<cpdr_fragment> frags;        // every fragment, segment-major order
    std::vector<int32_t> pre_items;          // fragments with CPDR_FRAG_CONT_NEXT
    std::vector<int32_t> fwd_order;          // fragments, longest first (fwd launch order)
    std::vector<MergeChain> chains;          // sequences spanning >= 2 segments
    std::vector<int32_t> zero_pre;           // segment indices with no continuing fragment
    std::vector<int32_t> zero_init;          // segment indices whose S_init is zero
    std::vector<int32_t> empty_seqs;         // zero-length sequences (final state = 0)
    int32_t max_pre_chunks = 0, max_fwd_chunks = 0;
    std::vector<int32_t> frag_chunk0;        // first global chunk of each fragment (+ total)
    std::vector<WyChunk> wy_chunks;          // every chunk of every fragment
    // host-buffer path: fragments in kHostParts groups of consecutive memory
    // tokens, so that the forward of a group can start once its q is in and
    // its o can leave while the next group runs
    std::vector<int32_t> bwd_pre_items;      // fragments continuing a sequence (backward pre-process)
    std::vector<int32_t> host_items;         // fragments, group by group (longest first inside)
    int32_t host_part_off[kHostParts + 1] = {};   // group g: host_items[off[g] .. off[g+1])
    int64_t host_part_tok[kHostParts + 1] = {};   // group g: memory tokens [tok[g], tok[g+1])
    int32_t conv_width = 0;                  // causal conv1d kernel size (0: no conv path)
    std::vector<ConvTile> conv_tiles;        // conv work units, fragment by fragment
    std::vector<int64_t> conv_halo;          // halo rows, conv_width - 1 memory positions each
    std::vector<int32_t> conv_pre_tokens;    // per segment: halo tokens inside its first sequence

    int32_t nseg() const { return R * B; }
};

// Builds the plan; returns CPDR_OK or an error with `err` set.
cpdr_status build_plan(const cpdr_desc &d, Plan &p, std::string &err);

// Device copies of the plan tables.
struct DeviceTables {
    cpdr_fragment *frags = nullptr;
    int32_t *pre_items = nullptr;
    int32_t *fwd_order = nullptr;
    MergeChain *chains = nullptr;
    int32_t *zero_pre = nullptr;
    int32_t *zero_init = nullptr;
    int32_t *empty_seqs = nullptr;
    int32_t *frag_chunk0 = nullptr;
    WyChunk *wy_chunks = nullptr;
    ConvTile *conv_tiles = nullptr;
    int32_t *host_items = nullptr;
    int32_t *bwd_pre_items = nullptr;
    int64_t *conv_halo = nullptr;
    int32_t *status = nullptr;   // device status word (bounded waits)
};

}  // namespace cpdr

struct cpdr_ctx {
    // The plan is built once and never changed afterwards; a copy of the
    // context (the allocation-free entry point's view with its own device
    // tables) shares it without copying it.
    std::shared_ptr<const cpdr::Plan> plan_store;
    const cpdr::Plan &plan;
    explicit cpdr_ctx(std::shared_ptr<const cpdr::Plan> p) : plan_store(std::move(p)), plan(*plan_store) {}
    cpdr::DeviceTables dev;
    bool has_device = false;
    bool use_tc = false;        // tcgen05 kernels for the bf16, d = 128 path
    int device = -1;
    // host-buffer path: a copy stream for the host-to-device copies and the
    // events that let compute start on the inputs that have arrived
    void *copy_stream = nullptr, *out_stream = nullptr;
    static constexpr int kHostEvents = 4 + 2 * cpdr::kHostParts;   // start, in0, in1, out, q[g], f[g]
    void *host_ev[kHostEvents] = {};
};

namespace cpdr {

// Launchers (kernels live in the .cu files).  Each returns a CUDA error code
// (0 = success) of the launch it enqueued.
int launch_simt_pre(const cpdr_ctx *c, const void *k, const void *v, const void *beta,
                    const float *g, float *S_ext, float *M, void *stream);
// items: fragment indices to run (n_items of them); the plan's fwd_order for all
int launch_simt_fwd(const cpdr_ctx *c, const int32_t *items, int n_items, const void *q, const void *k, const void *v,
                    const void *beta, const float *g, const float *S_init, void *o,
                    float *final_state, void *stream);
int launch_merge(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init,
                 void *stream);
// The merge on the tensor cores (tc_merge.cu; bf16 hi/lo splits, d = 128).
int launch_tc_merge(const cpdr_ctx *c, const float *S_ext, const float *M, float *S_init, void *stream);
// The backward's reverse merge G <- M_j^T G + dS_ext[j] on the tensor cores.
int launch_tc_merge_rev(const cpdr_ctx *c, const float *dS_ext, const float *M, float *dS_end, void *stream);
int launch_zero_segments(const cpdr_ctx *c, float *S_ext, float *M, float *S_init,
                         float *final_state, int which, void *stream);
// True when the tcgen05 kernels cover this problem (bf16, dk = dv = 128, scalar gate).
bool tc_supported(const Plan &p);

// Status word of the allocation-free entry point's device array on device
// `dev` (noalloc.cu); nullptr until that entry point has been set up there.
int32_t *noalloc_status_word(int dev);

// Sets this thread's last-error message and returns the status.
cpdr_status fail_with(cpdr_status s, const std::string &msg);

// Number of kernels one preprocess + merge + fwd step enqueues (final_state given).
int launches_per_step(const cpdr_ctx *c);

// Bytes of the WY tile workspace (0 when the CUDA-core kernels are used).
size_t wy_bytes(const cpdr_ctx *c);

int launch_tc_kda_prep(const cpdr_ctx *c, const void *k, const void *q, const void *beta, const float *g,
                       void *wy, void *stream);
// The same, also writing T of every unit as fp32 64 x 64 into tmat (the backward).
int launch_tc_kda_prep_t(const cpdr_ctx *c, const void *k, const void *q, const void *beta, const float *g,
                         void *wy, float *tmat, void *stream);
int launch_tc_wy(const cpdr_ctx *c, const void *k, const void *beta, const float *g, void *wy,
                 void *stream);
// The same, also writing T of every unit as fp32 64 x 64 into tmat (the backward).
int launch_tc_wy_t(const cpdr_ctx *c, const void *k, const void *beta, const float *g, void *wy, float *tmat,
                   void *stream);
int launch_tc_pre(const cpdr_ctx *c, const void *k, const void *v, const float *g, const void *wy,
                  float *S_ext, float *M, void *stream);
// Backward on the tensor cores (tc_chain.cu): the forward recomputation
// storing each chunk's starting state and Delta, and the state-gradient
// chains (pre-process of the backward, main pass).
int launch_tc_rec(const cpdr_ctx *c, const void *k, const void *v, const float *g, const void *wy,
                  const float *S_init, float *st_S, float *st_D, void *stream);
int launch_tc_bwd_chain(const cpdr_ctx *c, const int32_t *items, int n_items, int pre, int gq, const void *q,
                        const void *k, const void *dout, const float *g, const void *wy, const float *dht,
                        const float *dS_end, float *dS_ext, float *st_dS, float *st_dD, void *stream);
// Input gradients per (chunk, head) from the recomputed states and the
// state-gradient chain's outputs (bwd_grad.cu).
int launch_bwd_grad(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta,
                    const float *g, const void *dout, const float *tmat, const float *st_S, const float *st_D,
                    const float *st_dS, const float *st_dD, float *dq, float *dk, float *dv, float *dbeta, float *dg,
                    void *stream);
// The same for the per-dim gate (bwd_grad_kda.cu): T from the preparation.
int launch_bwd_grad_kda(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta,
                        const float *g, const void *dout, const float *tmat, const float *st_S, const float *st_D,
                        const float *st_dS, const float *st_dD, float *dq, float *dk, float *dv, float *dbeta,
                        float *dg, void *stream);
// The backward runs on the tensor cores (bf16, d = 128, scalar gate, Hq == H,
// [dk, dv] states); its scratch bytes (bwd.cu).
bool bwd_simt_fits(const cpdr_ctx *c);
bool bwd_uses_tc(const cpdr_ctx *c);
size_t bwd_tc_scratch_bytes(const cpdr_ctx *c);
// Backward (bwd.cu): scratch per CTA and the grid it is sized for.
size_t bwd_scratch_floats_per_cta(const cpdr_ctx *c);
int bwd_grid(const cpdr_ctx *c);
int launch_bwd(const cpdr_ctx *c, const void *q, const void *k, const void *v, const void *beta, const float *g,
               const void *dout, const float *dht, const float *S_init, const float *M, float *dS_ext,
               float *dS_end, float *scratch, float *dq, float *dk, float *dv, float *dbeta, float *dg,
               void *stream);
int launch_conv1d(const cpdr_ctx *c, const void *x, const float *weight, const float *bias, int channels,
                  int activation, void *y, void *stream);
int launch_tc_fwd(const cpdr_ctx *c, const int32_t *items, int n_items, const void *q, const void *k, const void *v,
                  const float *g,
                  const void *wy, const float *S_init, void *o, float *final_state, void *stream);

}  // namespace cpdr
