// route_noalloc.cu -- sse_route_noalloc: the router and token->partition
// grouping of sse_route for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin running inside a
// host application that owns every device allocation and hands out only the
// tensors it manages, a serving loop that must never pay the device-wide
// synchronisation a cudaMalloc can cause, or code written in a language with
// no binding to the CUDA allocator.  This entry point needs only the caller's
// inputs and outputs; the routing stage's scratch (per-sequence block
// prefixes and per-block partition counts) lives in a fixed array that is
// part of the library's own device image.
//
// That array exists once on every GPU that loads the library and stays
// reserved there until the process exits.  All calls on a device share it,
// and it keeps whatever the previous call left: nothing in it has to start
// at zero, because each call writes every entry it reads before reading it.
// Two calls whose kernels overlap on the same GPU (different streams, or
// different host threads) race on the array and corrupt each other's
// results; serialise them.
#include "sse_internal.cuh"

namespace {

// 4 MiB: room for (num_seqs + 1) + 4 * B + H * N * (B + 1) int32 entries,
// B = ceil(T / 256) + num_seqs routing blocks, plus the 256-byte alignment of
// the three regions; with 16 heads and 16 partitions that is about one
// million tokens per call.
constexpr size_t kScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

// Device address of g_route_scratch in the current device's context.  In
// host code the array's name is only a host-side stand-in, so the address is
// looked up through the runtime, with the device current, on every call: the
// lookup is a cheap host-side query, and a cached address could outlive its
// context (after cudaDeviceReset, or for a caller on another context of the
// same device).
cudaError_t scratch_address(void **addr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    *addr = p;
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" sse_status_t sse_route_noalloc(const sse_config_t *cfg, const void *router_logits,
                                          const int32_t *cu_seqlens, int32_t num_seqs,
                                          int64_t total_tokens, int32_t *topk_idx, float *topk_w,
                                          int32_t *seg_off, int32_t *perm, sse_stream_t stream) {
    // Argument checks: the same rules (and the same code) as sse_route, minus
    // the workspace.
    sse_status_t st = sse::check_config(cfg);
    if (st != SSE_OK) return st;
    const sse_config_t &c = *cfg;
    if ((st = sse::check_sizes(c, total_tokens, num_seqs)) != SSE_OK) return st;
    if (!cu_seqlens || !topk_idx || (total_tokens > 0 && !router_logits)) return SSE_ERR_INVALID_ARG;
    if (!aligned16(router_logits)) return SSE_ERR_INVALID_ARG;
    const bool group = seg_off || perm;
    if (group && !(seg_off && perm)) return SSE_ERR_INVALID_ARG;

    // Scratch layout and the size limit, checked before any CUDA call.
    const int64_t max_blocks = sse::route_max_blocks(total_tokens, num_seqs);
    const int64_t cnt_entries = (int64_t)c.num_heads * c.num_partitions * (max_blocks + 1);
    sse::Carver cv(nullptr);
    cv.take<int32_t>((size_t)num_seqs + 1);
    cv.take<int4>((size_t)max_blocks);
    cv.take<int32_t>((size_t)cnt_entries);
    if (cv.off > kScratchBytes) return SSE_ERR_WORKSPACE;
    if (num_seqs == 0) return SSE_OK;

    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return SSE_ERR_CUDA;
    sse::Carver sc(scratch);
    sse::RouteBuffers rb{};
    rb.max_blocks = (int32_t)max_blocks;
    rb.blk_prefix = sc.take<int32_t>((size_t)num_seqs + 1);
    rb.blk_info = sc.take<int4>((size_t)max_blocks);
    rb.cnt = sc.take<int32_t>((size_t)cnt_entries);
    rb.seg_off = seg_off;
    rb.topk_idx = topk_idx;
    rb.topk_w = topk_w;
    rb.perm = perm;
    rb.perm_rec = nullptr;
    rb.perm_e = nullptr;
    cudaError_t e = sse::launch_route(c, router_logits, cu_seqlens, num_seqs, total_tokens, rb, group,
                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSE_OK : SSE_ERR_CUDA;
}
