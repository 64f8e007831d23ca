// sse_internal.cuh -- device helpers and launcher declarations shared by the
// translation units of libsse.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/sse.h"

namespace sse {

constexpr int kMaxPartitions = 64;
constexpr int kMaxTopK = 8;
constexpr int kMaxHeads = 1 << 16;  // bounds the size products of the host checks
constexpr int kMaxDim = 1 << 12;    // key_dim, value_dim
constexpr int kRouteBlock = 256;  // tokens per routing block (one thread per token)
constexpr int kRouteLaunches = 5; // kernels launch_route issues when grouping
constexpr int kChunkRows = 128;   // rows of a tensor-core chunk; output regions are padded to it

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The routing kernels after the first are
// launched so that each may start while the previous one in the stream is
// finishing (its CTAs are scheduled and run their prologue early).  (The
// forward's later kernels launch the ordinary way: as dependents they made
// the whole step 13 us slower.)  Every kernel of such a chain
// calls griddep_wait() before it touches global memory -- and before any
// early return, so that no grid of the chain completes before the one ahead
// of it -- and calls griddep_launch_dependents() at its start, which lets the
// next kernel be scheduled once all of this grid's CTAs are running.  Both are
// no-ops for a kernel launched the ordinary way.  What an earlier kernel of
// the chain wrote is read with coherent loads only: no const __restrict__
// pointer and no __ldg on it (the read-only cache path assumes data that does
// not change during the reading kernel's lifetime, and a dependent kernel's
// lifetime begins before its predecessor has finished writing).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Element access for the two storage dtypes.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
    // four consecutive elements (16-byte aligned for float)
    static __device__ __forceinline__ float4 load4(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ void store4(float *p, float4 x) {
        *reinterpret_cast<float4 *>(p) = x;
    }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) {
        *p = __float2bfloat16_rn(x);
    }
    // four consecutive elements (8-byte aligned)
    static __device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
        uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        float4 f;
        f.x = __uint_as_float(u.x << 16);
        f.y = __uint_as_float(u.x & 0xffff0000u);
        f.z = __uint_as_float(u.y << 16);
        f.w = __uint_as_float(u.y & 0xffff0000u);
        return f;
    }
    static __device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 x) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&lo);
        u.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(p) = u;
    }
};

// ---------------------------------------------------------------------------
// Router for one (token, head): softmax over N logits in fp32 and the top-k
// by logit, equal logits ordered by ascending index (strict comparison while
// scanning upward keeps the lower index).  idx/w receive k entries in
// descending-logit order.  NP >= N bounds the unrolled loops (8, 16, 32 or
// 64); `vec` says that the N logits of the row are 16-byte aligned and fill
// whole 16-byte words, so they are read with vector loads.
// ---------------------------------------------------------------------------
template <typename T, int NP>
__device__ __forceinline__ void route_token(const T *logit, int N, int k, bool vec, int *idx, float *w) {
    float l[NP];
    constexpr int EPV = 16 / sizeof(T);  // elements per 16-byte word
    if (vec) {
#pragma unroll
        for (int i0 = 0; i0 < NP; i0 += EPV) {
            if (i0 < N) {
                const uint4 u = __ldg(reinterpret_cast<const uint4 *>(logit + i0));
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (sizeof(T) == 2)
                        l[i0 + e] = __uint_as_float(e & 1 ? (wv[e / 2] & 0xffff0000u) : (wv[e / 2] << 16));
                    else
                        l[i0 + e] = __uint_as_float(wv[e]);
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < NP; ++i)
            if (i < N) l[i] = Elem<T>::load(logit + i);
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NP; ++i)
        if (i < N) m = fmaxf(m, l[i]);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NP; ++i)
        if (i < N) s += expf(l[i] - m);
    const float inv = 1.f / s;
    uint64_t taken = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        int bi = -1;
        float bv = -INFINITY;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            if (i < N && !((taken >> i) & 1ull) && (bi < 0 || l[i] > bv)) {
                bv = l[i];
                bi = i;
            }
        }
        taken |= 1ull << bi;
        idx[j] = bi;
        w[j] = expf(bv - m) * inv;
    }
}

// The same router evaluated by one warp (lane i holds logits i and i + 32):
// max, sum of exponentials and k rounds of argmax (ties -> lower index) by
// shuffles.  Every lane returns the full result.
template <typename T>
__device__ __forceinline__ void route_token_warp(const T *logit, int N, int k, int lane, int *idx, float *w) {
    const float l0 = lane < N ? Elem<T>::load(logit + lane) : -INFINITY;
    const float l1 = lane + 32 < N ? Elem<T>::load(logit + lane + 32) : -INFINITY;
    float m = fmaxf(l0, l1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = (lane < N ? expf(l0 - m) : 0.f) + (lane + 32 < N ? expf(l1 - m) : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.f / s;
    bool t0 = lane >= N, t1 = lane + 32 >= N;  // taken (or absent)
    for (int j = 0; j < k; ++j) {
        // this lane's best remaining candidate; the lower index wins ties
        float bv = -INFINITY;
        int bi = 1 << 30;
        if (!t0) { bv = l0; bi = lane; }
        if (!t1 && (bi == (1 << 30) || l1 > bv)) { bv = l1; bi = lane + 32; }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != (1 << 30) && (bi == (1 << 30) || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi == lane) t0 = true;
        if (bi == lane + 32) t1 = true;
        idx[j] = bi;
        w[j] = expf(bv - m) * inv;
    }
}

// ---------------------------------------------------------------------------
// Host-side argument checks shared by every entry point (sse_api.cu):
// check_config validates the configuration, check_sizes the token and
// sequence counts against the kernels' 32-bit row and record indices.
// ---------------------------------------------------------------------------
sse_status_t check_config(const sse_config_t *cfg);
sse_status_t check_sizes(const sse_config_t &c, int64_t total_tokens, int32_t num_seqs);

// ---------------------------------------------------------------------------
// Workspace carving (256-byte aligned regions).
// ---------------------------------------------------------------------------
struct Carver {
    uintptr_t base;
    size_t off = 0;
    explicit Carver(void *p) : base(reinterpret_cast<uintptr_t>(p)) {}
    template <typename T> T *take(size_t n) {
        off = (off + 255) & ~size_t(255);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += n * sizeof(T);
        return p;
    }
};

// Device buffers of the routing/grouping stage.
struct RouteBuffers {
    int32_t *blk_prefix;  // [num_seqs + 1] routing blocks before each sequence
    int4 *blk_info;       // [max_blocks] (sequence, first token, end token, 0) per block; sequence -1 past the last
    int32_t *cnt;         // [H * N * (max_blocks + 1)] per-block counts, scanned in place
    int32_t *seg_off;     // [num_seqs * H * N + 1]
    int32_t *topk_idx;    // [T * H * k]
    float *topk_w;        // [T * H * k]
    int32_t *perm;        // [H * k * T] token ids (may be null)
    int32_t *perm_rec;    // [H * k * T] record ids t * k + j (may be null)
    float *perm_e;        // [H * k * T] router weight of each record (may be null)
    // Output placement of the chunked forward (both may be null).  Work items
    // are the shared segments (b, h) first, then the routed segments s; item
    // u owns the partial-output rows pad_off[u] .. pad_off[u] + len_u, its
    // length rounded up to whole chunks (kChunkRows).
    int32_t *pad_off;     // [num_items + 1]
    int32_t *rec_pos;     // [T * H * (k + shared)] partial row of each contribution of (t, h)
    int32_t max_blocks;
};

int64_t route_max_blocks(int64_t total_tokens, int32_t num_seqs);

// Masking schedule (no grouping): the chunk-padded output region of every work
// item (shared (b, h), then (b, h, i) over whole sequences) and the partial row
// of each contribution of (t, h); needs topk_idx.  Two launches.
cudaError_t launch_masked_plan(const sse_config_t &cfg, const int32_t *cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, const RouteBuffers &rb, cudaStream_t stream);

// Launches the routing + grouping kernels; returns cudaGetLastError().
cudaError_t launch_route(const sse_config_t &cfg, const void *logits, const int32_t *cu_seqlens,
                         int32_t num_seqs, int64_t total_tokens, const RouteBuffers &rb,
                         bool group, cudaStream_t stream);

// Recurrent (CUDA-core) forward over all segments; writes fp32 partials that
// launch_combine sums.  The chunked path writes bf16 slots for launch_slot_combine.
struct ForwardArgs {
    const void *q, *k, *v, *g, *qs, *ks;
    const int32_t *cu_seqlens;
    int32_t num_seqs;
    int64_t total_tokens;
    const float *init;
    float *final_state;
    void *out;
    const int32_t *seg_off;
    const int32_t *perm_rec;
    const float *perm_e;
    const float *topk_w;
    const int32_t *topk_idx; // masking schedule: the selected partitions of each (t, h)
    const int32_t *pad_off;  // chunked path: first partial row of each work item
    const int32_t *rec_pos;  // chunked path: partial rows of each (t, h)
    int64_t part_rows;       // chunked path: rows of the partial buffer
    void *part_routed;   // recurrent: [T, H, k, d] fp32; chunked: [part_rows, d] bf16 in work-item order
    void *part_shared;   // recurrent: [T, H, d] fp32; chunked: unused
    int32_t part_bf16;
    int32_t *flags;      // [0]: device-check flags; [1]: entries of redo_list; [2]: chunked work counter
    void *chunk_ws;      // chunked path scratch
    int32_t *redo_list;  // chunked path: work items to recompute token by token
};

bool recurrent_supported(const sse_config_t &cfg);
cudaError_t launch_forward_recurrent(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream);

bool chunked_supported(const sse_config_t &cfg);
size_t chunked_extra_workspace(const sse_config_t &cfg, int64_t total_tokens, int32_t num_seqs);
// Adds the number of kernels it launched to *launches.
cudaError_t launch_forward_chunked(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream,
                                   int *launches);

// out[t,h,:] = sum_j part_routed[t,h,j,:] + part_shared[t,h,:]   (recurrent path)
cudaError_t launch_combine(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream);
// out[t,h,:] = sum over j of the bf16 partial row rec_pos[(t*H+h)*(k+shared)+j]   (chunked path)
cudaError_t launch_gather_combine(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream);
// Rows of the chunked path's partial buffer: every work item padded to whole chunks.
int64_t chunked_part_rows(const sse_config_t &cfg, int64_t total_tokens, int32_t num_seqs);

// Backward (backward.cu): pointers as in sse_backward, plus the routing of
// the forward (recomputed) and the contribution slots [T, H, k + shared, width]
// of every (token, head) that the combine pass sums.
struct BackwardArgs {
    const void *q, *k, *v, *g, *logits, *qs, *ks, *d_out;
    const int32_t *cu_seqlens;
    int32_t num_seqs;
    int64_t total_tokens;
    const float *init, *d_final;
    void *dq, *dk, *dv, *dg, *d_logits, *dq_shared, *dk_shared;
    float *d_init;
    const int32_t *seg_off, *perm_rec, *topk_idx;
    const float *perm_e;
    // contribution slots: dq, dk and dv in the I/O type (each a single product
    // or sum, rounded once), dg in float32 (it holds reverse running sums)
    void *dq_c, *dk_c, *dv_c;
    float *dg_c;
    float *de_c;                       // [T, H, k, 2] router-weight gradient of each selected partition (read, write)
    // Per-token kernel restricted to a list of work items (shared (b, h) first,
    // then routed (b, h, i)): item seg_list[x] for x < *seg_count.  Null: all.
    const int32_t *seg_list, *seg_count;
    // Chunked (tensor-core) form, c = 128: buffers of backward_chunked.cu.
    const int32_t *pad_off;  // chunk-padded first row of each work item; chunk = row / 128
    int64_t num_chunks;      // upper bound of the chunks (launch size; items past the last exit)
    __nv_bfloat16 *ustate;   // [chunks, c, d]: K_hat^T V of the chunk (bf16; the scan sums in fp32)
    __nv_bfloat16 *wgrad;    // [chunks, c, d]: Q_hat^T dO of the chunk (likewise)
    float *gamma;            // [chunks, c]: exp(G_last), the chunk's decay of each state row
    float *gml;              // [chunks, 2, c]: G_m and G_l of each state row
    void *sp_tiles;          // [chunks, 32 KB]: S' = diag(exp(G_m)) S_start, bf16 in the operand tile layout
    void *dsp_tiles;         // [chunks, 32 KB]: dS' = diag(exp(G_l - G_m)) dS_end, likewise
    float *gscratch;         // [kBwdScratchCtas, 128, c]: G_r - G_m of the chunk in flight, per CTA
    float *fterm;            // [items, c]: rowsum(S_T * dL/dS_T) of each work item
    float *dgtot;            // [chunks, c]: gate-gradient column totals of each chunk
    int32_t *marks;          // [items]: item queued for the per-token kernel (gate range)
    int32_t *redo_list;      // [items] and its length in flags[1]
    int32_t *flags;          // [0]: device-check flags, [1]: entries of redo_list
};
constexpr int kBwdScratchCtas = 256;  // CTAs of the chunked gradient kernel (one scratch slot each)
bool backward_supported(const sse_config_t &cfg);
// The chunked form: bf16, c = 128, d in {64, 128}.
bool backward_chunked_supported(const sse_config_t &cfg);
// Launches the chunked form: every work item, then the per-token kernel over
// the items whose gates left the factorised form's range, then the per-token
// sums.  Adds the number of kernels it launched to *launches.
cudaError_t launch_backward_chunked(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream,
                                    int *launches);
// The per-token kernel over the items a.seg_list names (all when null).
cudaError_t launch_backward_segments(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream);
cudaError_t launch_backward_combine(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream);
// Adds the number of kernels it launched to *launches.
cudaError_t launch_backward(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream, int *launches);

// SSE on a gated delta-rule transition (delta.cu).  log_alpha, beta:
// [T, H] in the token dtype.  Forward read-outs go to the float32 partial
// slots of the recurrent path (part_routed [T, H, k, d], part_shared
// [T, H, d]) that launch_combine sums.
struct DeltaArgs {
    const void *q, *k, *v, *log_alpha, *beta, *qs, *ks;
    const int32_t *cu_seqlens;
    int32_t num_seqs;
    int64_t total_tokens;
    const float *init;
    float *final_state;
    const int32_t *seg_off, *perm_rec;
    const float *topk_w;
    float *part_routed, *part_shared;
    int32_t *flags;  // status words of the chunked form: [0] device flags, [1] work counter
};
struct DeltaDecodeArgs {
    const void *q, *k, *v, *log_alpha, *beta, *logits, *qs, *ks;
    int32_t batch;
    float *state;
    void *out;
    int32_t *topk_idx;
    float *topk_w;
};
bool delta_supported(const sse_config_t &cfg);
cudaError_t launch_delta_forward(const sse_config_t &cfg, const DeltaArgs &a, cudaStream_t stream);
// Chunked delta-rule forward on the tensor cores (delta_chunked.cu): bf16, c = d = 128.
bool delta_chunked_supported(const sse_config_t &cfg);
cudaError_t launch_delta_chunked(const sse_config_t &cfg, const DeltaArgs &a, cudaStream_t stream);
// Whether sse_delta_forward takes the chunked form (which writes bf16 partial rows).
inline bool delta_chunked_partials_bf16(const sse_config_t &cfg) {
    return cfg.algo != SSE_ALGO_RECURRENT && delta_chunked_supported(cfg);
}
cudaError_t launch_delta_decode(const sse_config_t &cfg, const DeltaDecodeArgs &a, cudaStream_t stream);

bool decode_supported(const sse_config_t &cfg);
cudaError_t launch_decode(const sse_config_t &cfg, const void *q, const void *k, const void *v,
                          const void *g, const void *logits, const void *qs, const void *ks,
                          int32_t batch, float *state, void *out, int32_t *topk_idx,
                          float *topk_w, cudaStream_t stream);

// Front end (projections from the hidden states); pointers as in sse_front_end.
struct FrontEndArgs {
    int64_t T;
    int32_t hidden;
    float gate_inv_tau;
    const void *x, *w_q, *w_k, *w_v, *w_g, *w_e, *a_q, *b_q, *a_k, *b_k;
    void *q, *k, *v, *g, *logits, *q_shared, *k_shared;
    void *xa;        // [T, 128] bf16 scratch: x A_q | x A_k
    int32_t *flags;
};
constexpr int kLoraRank = 64;
bool front_end_supported(const sse_config_t &cfg, int32_t hidden);
// Adds the number of kernels it launched to *launches.
cudaError_t launch_front_end(const sse_config_t &cfg, const FrontEndArgs &f, cudaStream_t stream, int *launches);

}  // namespace sse
