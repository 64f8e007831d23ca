// sse_api.cu -- the extern "C" entry points of libsse (declared and
// documented in include/sse.h): host-side validation, workspace layout and
// the launch sequence of each call.  No allocation, no synchronization
// (except sse_read_device_status).
#include <algorithm>
#include <cmath>
#include <initializer_list>

#include "sse_internal.cuh"

#ifdef SSE_NVTX
#include <nvtx3/nvToolsExt.h>
// One NVTX range per entry-point call, for profiler timelines; compiled in
// only with -DSSE_NVTX (build.py: SSE_NVTX=1 in the environment).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};
#define SSE_RANGE(name) NvtxRange sse_nvtx_range_(name)
#else
#define SSE_RANGE(name) ((void)0)
#endif

namespace sse {

namespace {
int elem_bytes(const sse_config_t &c) { return c.dtype == SSE_BF16 ? 2 : 4; }
}  // namespace

sse_status_t check_config(const sse_config_t *cfg) {
    if (!cfg) return SSE_ERR_INVALID_ARG;
    const sse_config_t &c = *cfg;
    if (c.num_heads < 1 || c.key_dim < 1 || c.value_dim < 1) return SSE_ERR_INVALID_ARG;
    if (c.num_partitions < 1 || c.top_k < 1 || c.top_k > c.num_partitions) return SSE_ERR_INVALID_ARG;
    if (c.use_shared != 0 && c.use_shared != 1) return SSE_ERR_INVALID_ARG;
    if (c.dtype != SSE_F32 && c.dtype != SSE_BF16) return SSE_ERR_INVALID_ARG;
    if (c.algo < SSE_ALGO_AUTO || c.algo > SSE_ALGO_MASKED) return SSE_ERR_INVALID_ARG;
    if (!std::isfinite(c.scale)) return SSE_ERR_INVALID_ARG;
    if (c.num_partitions > kMaxPartitions || c.top_k > kMaxTopK) return SSE_ERR_UNSUPPORTED;
    if (c.num_heads > kMaxHeads || c.key_dim > kMaxDim || c.value_dim > kMaxDim) return SSE_ERR_UNSUPPORTED;
    if ((c.key_dim * elem_bytes(c)) % 16 || (c.value_dim * elem_bytes(c)) % 16) return SSE_ERR_UNSUPPORTED;
    return SSE_OK;
}

sse_status_t check_sizes(const sse_config_t &c, int64_t total_tokens, int32_t num_seqs) {
    if (num_seqs < 0 || total_tokens < 0) return SSE_ERR_INVALID_ARG;
    if (num_seqs == 0 && total_tokens != 0) return SSE_ERR_INVALID_ARG;
    // Bound each factor before forming a product: with total_tokens < 2^31,
    // heads <= kMaxHeads and top_k <= kMaxTopK every product below fits in
    // 64 bits.
    if (total_tokens >= (int64_t(1) << 31)) return SSE_ERR_UNSUPPORTED;
    const int64_t recs = total_tokens * c.num_heads * c.top_k;
    if (recs >= (int64_t(1) << 31) || total_tokens * c.top_k >= (int64_t(1) << 31)) return SSE_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * c.num_heads * c.num_partitions >= (int64_t(1) << 30)) return SSE_ERR_UNSUPPORTED;
    if (chunked_part_rows(c, total_tokens, num_seqs) >= (int64_t(1) << 31)) return SSE_ERR_UNSUPPORTED;
    return SSE_OK;
}

}  // namespace sse

namespace {

using sse::Carver;
using sse::RouteBuffers;
using sse::check_config;
using sse::check_sizes;

constexpr int32_t kAbiVersion = 2;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Route-stage buffers carved from the workspace.  User-provided outputs are
// used in place; missing ones live in the workspace.
RouteBuffers carve_route(Carver &cv, const sse_config_t &c, int64_t T, int32_t S, int32_t *topk_idx,
                         float *topk_w, int32_t *seg_off, int32_t *perm, bool need_w, bool need_rec,
                         bool need_pos = false) {
    RouteBuffers rb{};
    rb.max_blocks = (int32_t)sse::route_max_blocks(T, S);
    rb.blk_prefix = cv.take<int32_t>(S + 1);
    rb.blk_info = cv.take<int4>((size_t)rb.max_blocks);
    rb.cnt = cv.take<int32_t>((size_t)c.num_heads * c.num_partitions * (rb.max_blocks + 1));
    int32_t *ws_seg = cv.take<int32_t>((size_t)S * c.num_heads * c.num_partitions + 1);
    int32_t *ws_idx = cv.take<int32_t>((size_t)T * c.num_heads * c.top_k);
    float *ws_w = need_w ? cv.take<float>((size_t)T * c.num_heads * c.top_k) : nullptr;
    int32_t *ws_rec = need_rec ? cv.take<int32_t>((size_t)T * c.num_heads * c.top_k) : nullptr;
    float *ws_pe = need_rec ? cv.take<float>((size_t)T * c.num_heads * c.top_k) : nullptr;
    rb.seg_off = seg_off ? seg_off : ws_seg;
    rb.topk_idx = topk_idx ? topk_idx : ws_idx;
    rb.topk_w = topk_w ? topk_w : ws_w;
    rb.perm = perm;
    rb.perm_rec = ws_rec;
    rb.perm_e = ws_pe;
    const int64_t nitems = (int64_t)S * c.num_heads * (c.num_partitions + c.use_shared);
    rb.pad_off = need_pos ? cv.take<int32_t>(nitems + 1) : nullptr;
    rb.rec_pos = need_pos ? cv.take<int32_t>((size_t)T * c.num_heads * (c.top_k + c.use_shared)) : nullptr;
    return rb;
}

bool use_chunked(const sse_config_t &c) {
    if (c.algo == SSE_ALGO_RECURRENT) return false;
    if (c.algo == SSE_ALGO_CHUNKED || c.algo == SSE_ALGO_MASKED) return true;
    return sse::chunked_supported(c);
}

// The concrete algorithm AUTO stands for (a pure function of the
// configuration, so the workspace size and the call agree): the grouped
// varlen schedule wherever the tensor-core path applies, else the recurrent
// path.  The pages ("Scaling Linear Attention with Sparse State Expansion",
// section 2.6) name masking for short inputs; on GB300 it was slower in every
// measured case, short ones and top_k == N (identity grouping) included --
// B2 T2048 H4 c=d=64 N8 k2: 0.109 ms masked vs 0.092 ms grouped; the same
// with N = k = 4: 0.131 vs 0.093 ms; B8 T4096 H16 c=d=128 N8 k2 with skewed
// loads: 1.53 vs 0.63 ms -- so AUTO never picks it.
sse_config_t resolve_algo(const sse_config_t &c, int64_t /*total_tokens*/, int32_t /*num_seqs*/) {
    sse_config_t r = c;
    if (c.algo == SSE_ALGO_AUTO) r.algo = sse::chunked_supported(c) ? SSE_ALGO_CHUNKED : SSE_ALGO_RECURRENT;
    return r;
}

struct ForwardLayout {
    RouteBuffers rb;
    void *part_routed, *part_shared;
    int64_t part_rows;
    int32_t *flags;
    void *chunk_ws;
    size_t bytes;
};

ForwardLayout carve_forward(void *ws, const sse_config_t &c, int64_t T, int32_t S,
                            int32_t *topk_idx, float *topk_w) {
    Carver cv(ws);
    ForwardLayout L{};
    L.flags = cv.take<int32_t>(64);
    const bool chunked = use_chunked(c);
    const bool masked = c.algo == SSE_ALGO_MASKED;  // no grouping: no per-record arrays
    L.rb = carve_route(cv, c, T, S, topk_idx, topk_w, nullptr, nullptr, true, !masked, chunked);
    if (chunked) {
        // bf16 partial read-outs, one row per contribution, in work-item order
        L.part_rows = sse::chunked_part_rows(c, T, S);
        L.part_routed = cv.take<unsigned char>((size_t)L.part_rows * c.value_dim * 2);
        L.part_shared = nullptr;
        L.chunk_ws = cv.take<unsigned char>(sse::chunked_extra_workspace(c, T, S));
    } else {
        // fp32 partial read-outs for the combine kernel
        L.part_routed = cv.take<float>((size_t)T * c.num_heads * c.top_k * c.value_dim);
        L.part_shared = c.use_shared ? cv.take<float>((size_t)T * c.num_heads * c.value_dim) : nullptr;
        L.chunk_ws = nullptr;
    }
    L.bytes = (cv.off + 255) & ~size_t(255);
    return L;
}

}  // namespace

extern "C" {

int32_t sse_abi_version(void) { return kAbiVersion; }

const char *sse_status_string(sse_status_t s) {
    switch (s) {
    case SSE_OK: return "SSE_OK";
    case SSE_ERR_INVALID_ARG: return "SSE_ERR_INVALID_ARG: invalid argument";
    case SSE_ERR_UNSUPPORTED: return "SSE_ERR_UNSUPPORTED: configuration not supported";
    case SSE_ERR_WORKSPACE: return "SSE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SSE_ERR_CUDA: return "SSE_ERR_CUDA: kernel launch failed";
    case SSE_ERR_DEVICE: return "SSE_ERR_DEVICE: a device-side check failed";
    case SSE_ERR_DEVICE_TIMEOUT: return "SSE_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel expired";
    default: return "unknown sse_status_t";
    }
}

size_t sse_route_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs) {
    if (check_config(cfg) != SSE_OK || check_sizes(*cfg, total_tokens, num_seqs) != SSE_OK) return 0;
    Carver cv(nullptr);
    carve_route(cv, *cfg, total_tokens, num_seqs, nullptr, nullptr, nullptr, nullptr, true, false);
    return (cv.off + 255) & ~size_t(255);
}

sse_status_t sse_route(const sse_config_t *cfg, const void *router_logits, const int32_t *cu_seqlens,
                       int32_t num_seqs, int64_t total_tokens, int32_t *topk_idx, float *topk_w,
                       int32_t *seg_off, int32_t *perm, void *workspace, size_t workspace_bytes,
                       sse_stream_t stream) {
    SSE_RANGE("sse_route");
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    if ((st = check_sizes(*cfg, total_tokens, num_seqs)) != SSE_OK) return st;
    if (!cu_seqlens || !topk_idx || (total_tokens > 0 && !router_logits)) return SSE_ERR_INVALID_ARG;
    if (!aligned16(router_logits)) return SSE_ERR_INVALID_ARG;
    const bool group = seg_off || perm;
    if (group && !(seg_off && perm)) return SSE_ERR_INVALID_ARG;
    const size_t need = sse_route_workspace_size(cfg, total_tokens, num_seqs);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return SSE_ERR_WORKSPACE;
    if (num_seqs == 0) return SSE_OK;
    Carver cv(workspace);
    RouteBuffers rb = carve_route(cv, *cfg, total_tokens, num_seqs, topk_idx, topk_w, seg_off, perm,
                                  true, false);
    cudaError_t e = sse::launch_route(*cfg, router_logits, cu_seqlens, num_seqs, total_tokens, rb,
                                      group, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
}

size_t sse_forward_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs) {
    if (check_config(cfg) != SSE_OK) return 0;
    const sse_config_t c = resolve_algo(*cfg, total_tokens, num_seqs);
    if (check_sizes(c, total_tokens, num_seqs) != SSE_OK) return 0;
    return carve_forward(nullptr, c, total_tokens, num_seqs, nullptr, nullptr).bytes;
}

sse_status_t sse_forward_timed(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                               const void *log_gate, const void *router_logits, const void *q_shared,
                               const void *k_shared, const int32_t *cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, const float *initial_state, float *final_state,
                               void *out, int32_t *topk_idx, float *topk_w, void *workspace,
                               size_t workspace_bytes, sse_stream_t stream, void *const *stage_events,
                               int32_t *num_launches) {
    SSE_RANGE("sse_forward_timed");
    if (num_launches) *num_launches = 0;
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    const sse_config_t c = resolve_algo(*cfg, total_tokens, num_seqs);
    if ((st = check_sizes(c, total_tokens, num_seqs)) != SSE_OK) return st;
    if (!cu_seqlens) return SSE_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !log_gate || !router_logits || !out))
        return SSE_ERR_INVALID_ARG;
    for (const void *p : std::initializer_list<const void *>{q, k, v, log_gate, router_logits, q_shared,
                                                             k_shared, out, (const void *)initial_state,
                                                             (const void *)final_state})
        if (!aligned16(p)) return SSE_ERR_INVALID_ARG;
    if (use_chunked(c)) {
        if (!sse::chunked_supported(c)) return SSE_ERR_UNSUPPORTED;
        if (c.algo == SSE_ALGO_MASKED && num_seqs > 12000) return SSE_ERR_UNSUPPORTED;
    } else if (!sse::recurrent_supported(c)) {
        return SSE_ERR_UNSUPPORTED;
    }
    const size_t need = sse_forward_workspace_size(cfg, total_tokens, num_seqs);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return SSE_ERR_WORKSPACE;
    if (num_seqs == 0) return SSE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto mark = [&](int i) {
        return stage_events ? cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s) : cudaSuccess;
    };
    ForwardLayout L = carve_forward(workspace, c, total_tokens, num_seqs, topk_idx, topk_w);
    if (mark(0) != cudaSuccess) return SSE_ERR_CUDA;
    if (cudaMemsetAsync(L.flags, 0, 64 * sizeof(int32_t), s) != cudaSuccess) return SSE_ERR_CUDA;
    const bool masked = c.algo == SSE_ALGO_MASKED;
    cudaError_t e = sse::launch_route(c, router_logits, cu_seqlens, num_seqs, total_tokens, L.rb, !masked, s);
    if (e != cudaSuccess) return SSE_ERR_CUDA;
    int launches = masked ? 2 : sse::kRouteLaunches;
    if (masked) {  // output placement of the masking schedule
        e = sse::launch_masked_plan(c, cu_seqlens, num_seqs, total_tokens, L.rb, s);
        if (e != cudaSuccess) return SSE_ERR_CUDA;
        launches += total_tokens > 0 ? 2 : 1;
    }
    if (mark(1) != cudaSuccess) return SSE_ERR_CUDA;
    sse::ForwardArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = log_gate; a.qs = q_shared; a.ks = k_shared;
    a.cu_seqlens = cu_seqlens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.init = initial_state;
    a.final_state = final_state;
    a.out = out;
    a.seg_off = L.rb.seg_off;
    a.perm_rec = L.rb.perm_rec;
    a.perm_e = L.rb.perm_e;
    a.topk_w = L.rb.topk_w;
    a.topk_idx = L.rb.topk_idx;
    a.pad_off = L.rb.pad_off;
    a.rec_pos = L.rb.rec_pos;
    a.part_rows = L.part_rows;
    a.part_routed = L.part_routed;
    a.part_shared = L.part_shared;
    a.part_bf16 = use_chunked(c) ? 1 : 0;
    a.flags = L.flags;
    a.chunk_ws = L.chunk_ws;
    a.redo_list = L.chunk_ws ? reinterpret_cast<int32_t *>(static_cast<unsigned char *>(L.chunk_ws) + 256) : nullptr;
    if (use_chunked(c)) {
        e = sse::launch_forward_chunked(c, a, s, &launches);
        if (e != cudaSuccess || mark(2) != cudaSuccess) return SSE_ERR_CUDA;
        e = sse::launch_gather_combine(c, a, s);
        launches += 1;
        if (e != cudaSuccess) return SSE_ERR_CUDA;
    } else {
        e = sse::launch_forward_recurrent(c, a, s);
        launches += 1;
        if (e != cudaSuccess || mark(2) != cudaSuccess) return SSE_ERR_CUDA;
        e = sse::launch_combine(c, a, s);
        launches += 1;
        if (e != cudaSuccess) return SSE_ERR_CUDA;
    }
    if (mark(3) != cudaSuccess) return SSE_ERR_CUDA;
    if (num_launches) *num_launches = launches;
    return SSE_OK;
}

sse_status_t sse_forward(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                         const void *log_gate, const void *router_logits, const void *q_shared,
                         const void *k_shared, const int32_t *cu_seqlens, int32_t num_seqs,
                         int64_t total_tokens, const float *initial_state, float *final_state,
                         void *out, int32_t *topk_idx, float *topk_w, void *workspace,
                         size_t workspace_bytes, sse_stream_t stream) {
    SSE_RANGE("sse_forward");
    return sse_forward_timed(cfg, q, k, v, log_gate, router_logits, q_shared, k_shared, cu_seqlens,
                             num_seqs, total_tokens, initial_state, final_state, out, topk_idx, topk_w,
                             workspace, workspace_bytes, stream, nullptr, nullptr);
}

sse_status_t sse_decode_step(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                             const void *log_gate, const void *router_logits, const void *q_shared,
                             const void *k_shared, int32_t batch, float *state, void *out,
                             int32_t *topk_idx, float *topk_w, sse_stream_t stream) {
    SSE_RANGE("sse_decode_step");
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    if (batch < 0) return SSE_ERR_INVALID_ARG;
    if ((int64_t)batch * cfg->num_heads >= (int64_t(1) << 31)) return SSE_ERR_UNSUPPORTED;
    if (batch > 0 && (!q || !k || !v || !log_gate || !router_logits || !state || !out))
        return SSE_ERR_INVALID_ARG;
    for (const void *p : std::initializer_list<const void *>{q, k, v, log_gate, router_logits, q_shared, k_shared, out, (const void *)state})
        if (!aligned16(p)) return SSE_ERR_INVALID_ARG;
    if (!sse::decode_supported(*cfg)) return SSE_ERR_UNSUPPORTED;
    cudaError_t e = sse::launch_decode(*cfg, q, k, v, log_gate, router_logits, q_shared, k_shared,
                                       batch, state, out, topk_idx, topk_w,
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
}

namespace {
struct BackwardLayout {
    RouteBuffers rb;
    void *dq_c, *dk_c, *dv_c;  // I/O type
    float *dg_c, *de_c;
    // chunked form
    bool chunked;
    int64_t num_chunks;
    __nv_bfloat16 *ustate, *wgrad;
    float *gamma, *gml, *gscratch, *fterm, *dgtot;
    void *sp_tiles, *dsp_tiles;
    int32_t *marks, *redo_list;
    int32_t *flags;  // status words first (sse_read_device_status reads word 0), both forms
    size_t bytes;
};

// The chunked (tensor-core) backward unless the recurrent one is asked for.
bool use_chunked_backward(const sse_config_t &c) {
    return c.algo != SSE_ALGO_RECURRENT && sse::backward_chunked_supported(c);
}

BackwardLayout carve_backward(void *ws, const sse_config_t &c, int64_t T, int32_t S) {
    Carver cv(ws);
    BackwardLayout L{};
    L.flags = cv.take<int32_t>(64);
    L.chunked = use_chunked_backward(c);
    L.rb = carve_route(cv, c, T, S, nullptr, nullptr, nullptr, nullptr, true, true, L.chunked);
    if (L.chunked) {
        sse_config_t grouped = c;
        grouped.algo = SSE_ALGO_AUTO;  // chunk-padded grouped records, as the chunked forward lays them out
        L.num_chunks = sse::chunked_part_rows(grouped, T, S) / sse::kChunkRows;
        const size_t nch = (size_t)L.num_chunks, kc = (size_t)c.key_dim, dv = (size_t)c.value_dim;
        const size_t nitems = (size_t)S * c.num_heads * (c.num_partitions + c.use_shared);
        L.ustate = cv.take<__nv_bfloat16>(nch * kc * dv);
        L.wgrad = cv.take<__nv_bfloat16>(nch * kc * dv);
        L.gamma = cv.take<float>(nch * kc);
        L.gml = cv.take<float>(nch * 2 * kc);
        L.sp_tiles = cv.take<unsigned char>(nch * sse::kChunkRows * 256);  // one 128 x 128 bf16 tile per chunk
        L.dsp_tiles = cv.take<unsigned char>(nch * sse::kChunkRows * 256);
        L.dgtot = cv.take<float>(nch * kc);
        L.gscratch = cv.take<float>((size_t)sse::kBwdScratchCtas * sse::kChunkRows * kc);
        L.fterm = cv.take<float>(nitems * kc);
        L.marks = cv.take<int32_t>(nitems);
        L.redo_list = cv.take<int32_t>(nitems);
    }
    const size_t slots = (size_t)T * c.num_heads * (c.top_k + c.use_shared);
    const size_t esz = c.dtype == SSE_BF16 ? 2 : 4;
    L.dq_c = cv.take<unsigned char>(slots * c.key_dim * esz);
    L.dk_c = cv.take<unsigned char>(slots * c.key_dim * esz);
    L.dg_c = cv.take<float>(slots * c.key_dim);
    L.dv_c = cv.take<unsigned char>(slots * c.value_dim * esz);
    L.de_c = cv.take<float>((size_t)T * c.num_heads * c.top_k * 2);
    L.bytes = (cv.off + 255) & ~size_t(255);
    return L;
}
}  // namespace

size_t sse_backward_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs) {
    if (check_config(cfg) != SSE_OK || check_sizes(*cfg, total_tokens, num_seqs) != SSE_OK) return 0;
    return carve_backward(nullptr, *cfg, total_tokens, num_seqs).bytes;
}

sse_status_t sse_backward(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                          const void *log_gate, const void *router_logits, const void *q_shared,
                          const void *k_shared, const int32_t *cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, const float *initial_state, const void *d_out,
                          const float *d_final_state, void *dq, void *dk, void *dv, void *d_log_gate,
                          void *d_router_logits, void *dq_shared, void *dk_shared, float *d_initial_state,
                          void *workspace, size_t workspace_bytes, sse_stream_t stream) {
    SSE_RANGE("sse_backward");
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    if ((st = check_sizes(*cfg, total_tokens, num_seqs)) != SSE_OK) return st;
    const sse_config_t &c = *cfg;
    if (!cu_seqlens) return SSE_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !log_gate || !router_logits || !d_out || !dq || !dk || !dv ||
                             !d_log_gate || !d_router_logits))
        return SSE_ERR_INVALID_ARG;
    // separate shared q / k get their own gradient buffers (and only then)
    if ((q_shared != nullptr) != (dq_shared != nullptr) || (k_shared != nullptr) != (dk_shared != nullptr))
        return SSE_ERR_INVALID_ARG;
    for (const void *p : std::initializer_list<const void *>{q, k, v, log_gate, router_logits, q_shared, k_shared,
                                                             (const void *)initial_state, d_out,
                                                             (const void *)d_final_state, dq, dk, dv, d_log_gate,
                                                             d_router_logits, dq_shared, dk_shared,
                                                             (const void *)d_initial_state})
        if (!aligned16(p)) return SSE_ERR_INVALID_ARG;
    if (!sse::backward_supported(c)) return SSE_ERR_UNSUPPORTED;
    if (c.algo == SSE_ALGO_CHUNKED && !sse::backward_chunked_supported(c)) return SSE_ERR_UNSUPPORTED;
    const size_t need = sse_backward_workspace_size(cfg, total_tokens, num_seqs);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return SSE_ERR_WORKSPACE;
    if (num_seqs == 0) return SSE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    BackwardLayout L = carve_backward(workspace, c, total_tokens, num_seqs);
    if (cudaMemsetAsync(L.flags, 0, 64 * sizeof(int32_t), s) != cudaSuccess) return SSE_ERR_CUDA;
    cudaError_t e = sse::launch_route(c, router_logits, cu_seqlens, num_seqs, total_tokens, L.rb, true, s);
    if (e != cudaSuccess) return SSE_ERR_CUDA;
    sse::BackwardArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = log_gate; a.logits = router_logits;
    a.qs = c.use_shared ? q_shared : nullptr;
    a.ks = c.use_shared ? k_shared : nullptr;
    a.d_out = d_out;
    a.cu_seqlens = cu_seqlens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.init = initial_state;
    a.d_final = d_final_state;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = d_log_gate; a.d_logits = d_router_logits;
    a.dq_shared = dq_shared; a.dk_shared = dk_shared;
    a.d_init = d_initial_state;
    a.seg_off = L.rb.seg_off;
    a.perm_rec = L.rb.perm_rec;
    a.perm_e = L.rb.perm_e;
    a.topk_idx = L.rb.topk_idx;
    a.dq_c = L.dq_c; a.dk_c = L.dk_c; a.dg_c = L.dg_c; a.dv_c = L.dv_c; a.de_c = L.de_c;
    int launches = sse::kRouteLaunches;
    if (L.chunked) {
        a.pad_off = L.rb.pad_off;
        a.num_chunks = L.num_chunks;
        a.ustate = L.ustate; a.wgrad = L.wgrad; a.gamma = L.gamma; a.gml = L.gml; a.gscratch = L.gscratch;
        a.sp_tiles = L.sp_tiles; a.dsp_tiles = L.dsp_tiles;
        a.fterm = L.fterm; a.dgtot = L.dgtot; a.marks = L.marks; a.redo_list = L.redo_list; a.flags = L.flags;
        e = sse::launch_backward_chunked(c, a, s, &launches);
        return e == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
    }
    e = sse::launch_backward(c, a, s, &launches);
    return e == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
}

namespace {
struct DeltaLayout {
    int32_t *flags;  // status words first (sse_read_device_status reads word 0)
    RouteBuffers rb;
    float *part_routed, *part_shared;
    size_t bytes;
};

DeltaLayout carve_delta(void *ws, const sse_config_t &c, int64_t T, int32_t S, int32_t *topk_idx, float *topk_w) {
    Carver cv(ws);
    DeltaLayout L{};
    L.flags = cv.take<int32_t>(64);
    L.rb = carve_route(cv, c, T, S, topk_idx, topk_w, nullptr, nullptr, true, true);
    L.part_routed = cv.take<float>((size_t)T * c.num_heads * c.top_k * c.value_dim);
    L.part_shared = c.use_shared ? cv.take<float>((size_t)T * c.num_heads * c.value_dim) : nullptr;
    L.bytes = (cv.off + 255) & ~size_t(255);
    return L;
}
}  // namespace

size_t sse_delta_forward_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs) {
    if (check_config(cfg) != SSE_OK || check_sizes(*cfg, total_tokens, num_seqs) != SSE_OK) return 0;
    return carve_delta(nullptr, *cfg, total_tokens, num_seqs, nullptr, nullptr).bytes;
}

sse_status_t sse_delta_forward(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                               const void *log_alpha, const void *beta, const void *router_logits,
                               const void *q_shared, const void *k_shared, const int32_t *cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, const float *initial_state,
                               float *final_state, void *out, int32_t *topk_idx, float *topk_w, void *workspace,
                               size_t workspace_bytes, sse_stream_t stream) {
    SSE_RANGE("sse_delta_forward");
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    if ((st = check_sizes(*cfg, total_tokens, num_seqs)) != SSE_OK) return st;
    const sse_config_t &c = *cfg;
    if (!cu_seqlens) return SSE_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !router_logits || !out))
        return SSE_ERR_INVALID_ARG;
    for (const void *p : std::initializer_list<const void *>{q, k, v, log_alpha, beta, router_logits, q_shared,
                                                             k_shared, out, (const void *)initial_state,
                                                             (const void *)final_state})
        if (!aligned16(p)) return SSE_ERR_INVALID_ARG;
    if (!sse::delta_supported(c)) return SSE_ERR_UNSUPPORTED;
    const size_t need = sse_delta_forward_workspace_size(cfg, total_tokens, num_seqs);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return SSE_ERR_WORKSPACE;
    if (num_seqs == 0) return SSE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeltaLayout L = carve_delta(workspace, c, total_tokens, num_seqs, topk_idx, topk_w);
    cudaError_t e = sse::launch_route(c, router_logits, cu_seqlens, num_seqs, total_tokens, L.rb, true, s);
    if (e != cudaSuccess) return SSE_ERR_CUDA;
    sse::DeltaArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
    a.qs = c.use_shared ? q_shared : nullptr;
    a.ks = c.use_shared ? k_shared : nullptr;
    a.cu_seqlens = cu_seqlens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.init = initial_state;
    a.final_state = final_state;
    a.seg_off = L.rb.seg_off;
    a.perm_rec = L.rb.perm_rec;
    a.topk_w = L.rb.topk_w;
    a.part_routed = L.part_routed;
    a.part_shared = L.part_shared;
    a.flags = L.flags;
    if (sse::launch_delta_forward(c, a, s) != cudaSuccess) return SSE_ERR_CUDA;
    sse::ForwardArgs fa{};
    fa.total_tokens = total_tokens;
    fa.out = out;
    fa.part_routed = L.part_routed;
    fa.part_shared = L.part_shared;
    fa.part_bf16 = sse::delta_chunked_partials_bf16(c) ? 1 : 0;  // the chunked form writes bf16 partials
    return sse::launch_combine(c, fa, s) == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
}

sse_status_t sse_delta_decode_step(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                                   const void *log_alpha, const void *beta, const void *router_logits,
                                   const void *q_shared, const void *k_shared, int32_t batch, float *state,
                                   void *out, int32_t *topk_idx, float *topk_w, sse_stream_t stream) {
    SSE_RANGE("sse_delta_decode_step");
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    if (batch < 0) return SSE_ERR_INVALID_ARG;
    if ((int64_t)batch * cfg->num_heads >= (int64_t(1) << 31)) return SSE_ERR_UNSUPPORTED;
    if (batch > 0 && (!q || !k || !v || !log_alpha || !beta || !router_logits || !state || !out))
        return SSE_ERR_INVALID_ARG;
    for (const void *p : std::initializer_list<const void *>{q, k, v, log_alpha, beta, router_logits, q_shared,
                                                             k_shared, out, (const void *)state})
        if (!aligned16(p)) return SSE_ERR_INVALID_ARG;
    if (!sse::delta_supported(*cfg)) return SSE_ERR_UNSUPPORTED;
    sse::DeltaDecodeArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.logits = router_logits;
    a.qs = cfg->use_shared ? q_shared : nullptr;
    a.ks = cfg->use_shared ? k_shared : nullptr;
    a.batch = batch;
    a.state = state;
    a.out = out;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    return sse::launch_delta_decode(*cfg, a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SSE_OK
                                                                                                    : SSE_ERR_CUDA;
}

size_t sse_front_end_workspace_size(const sse_config_t *cfg, int32_t hidden, int64_t total_tokens) {
    if (!cfg || hidden < 0 || total_tokens < 0) return 0;
    Carver cv(nullptr);
    cv.take<int32_t>(64);                                          // device-check flags
    cv.take<uint16_t>((size_t)total_tokens * 2 * sse::kLoraRank);  // x A_q | x A_k, bf16
    return (cv.off + 255) & ~size_t(255);
}

sse_status_t sse_front_end(const sse_config_t *cfg, int32_t hidden, int64_t total_tokens, const void *x,
                           const void *w_q, const void *w_k, const void *w_v, const void *w_g,
                           const void *w_e, const void *a_q, const void *b_q, const void *a_k,
                           const void *b_k, float gate_inv_tau, void *q, void *k, void *v,
                           void *log_gate, void *router_logits, void *q_shared, void *k_shared,
                           void *workspace, size_t workspace_bytes, sse_stream_t stream) {
    SSE_RANGE("sse_front_end");
    sse_status_t st = check_config(cfg);
    if (st != SSE_OK) return st;
    if (hidden < 0 || total_tokens < 0 || !std::isfinite(gate_inv_tau)) return SSE_ERR_INVALID_ARG;
    if (!sse::front_end_supported(*cfg, hidden)) return SSE_ERR_UNSUPPORTED;
    // row tiles of 128 tokens; every tile index fits in 32 bits
    if (total_tokens > 0 && total_tokens < 128) return SSE_ERR_UNSUPPORTED;
    if (total_tokens / 128 * (4 * (int64_t)cfg->num_heads + 1) >= (int64_t(1) << 31)) return SSE_ERR_UNSUPPORTED;
    const bool lora = a_q || b_q || a_k || b_k;
    if (lora && !(a_q && b_q && a_k && b_k && q_shared && k_shared)) return SSE_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!x || !w_q || !w_k || !w_v || !w_g || !w_e || !q || !k || !v || !log_gate ||
                             !router_logits))
        return SSE_ERR_INVALID_ARG;
    for (const void *p : std::initializer_list<const void *>{x, w_q, w_k, w_v, w_g, w_e, a_q, b_q, a_k, b_k, q, k,
                                                             v, log_gate, router_logits, q_shared, k_shared})
        if (!aligned16(p)) return SSE_ERR_INVALID_ARG;
    const size_t need = sse_front_end_workspace_size(cfg, hidden, total_tokens);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return SSE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Carver cv(workspace);
    sse::FrontEndArgs f{};
    f.flags = cv.take<int32_t>(64);
    f.xa = cv.take<uint16_t>((size_t)total_tokens * 2 * sse::kLoraRank);
    if (cudaMemsetAsync(f.flags, 0, 64 * sizeof(int32_t), s) != cudaSuccess) return SSE_ERR_CUDA;
    f.T = total_tokens;
    f.hidden = hidden;
    f.gate_inv_tau = gate_inv_tau;
    f.x = x;
    f.w_q = w_q;
    f.w_k = w_k;
    f.w_v = w_v;
    f.w_g = w_g;
    f.w_e = w_e;
    f.a_q = lora ? a_q : nullptr;
    f.b_q = lora ? b_q : nullptr;
    f.a_k = lora ? a_k : nullptr;
    f.b_k = lora ? b_k : nullptr;
    f.q = q;
    f.k = k;
    f.v = v;
    f.g = log_gate;
    f.logits = router_logits;
    f.q_shared = lora ? q_shared : nullptr;
    f.k_shared = lora ? k_shared : nullptr;
    int launches = 0;
    return sse::launch_front_end(*cfg, f, s, &launches) == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
}

sse_status_t sse_read_device_status(void *workspace, int32_t *flags, sse_stream_t stream) {
    if (!workspace || !flags || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SSE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SSE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSE_ERR_CUDA;
    *flags = host;
    if (host & SSE_DEVICE_TIMEOUT) return SSE_ERR_DEVICE_TIMEOUT;
    if (host & ~SSE_DEVICE_RECOMPUTED) return SSE_ERR_DEVICE;
    return SSE_OK;
}

sse_status_t sse_get_last_device_error(void *workspace, sse_stream_t stream) {
    int32_t flags = 0;
    return sse_read_device_status(workspace, &flags, stream);
}

}  // extern "C"
