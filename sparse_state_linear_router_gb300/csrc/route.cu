// route.cu -- router (eqs. 9-10 of "Scaling Linear Attention with Sparse
// State Expansion") and the token->partition grouping of its varlen schedule
// (section 2.6): a stable counting sort of the routed records by segment
// s = (b*H + h)*N + i that keeps each segment in time order.
//
// Stages (all deterministic, integer-exact):
//   plan     1 CTA   : routing blocks per sequence (256 tokens, never
//                      straddling a sequence) -> blk_prefix, and the table
//                      blk_info (sequence, token range) of every block
//   count    (blk,H) : route every token of the block, write topk_idx/topk_w,
//                      per-block histogram over partitions -> cnt
//   scan     (H*N)   : exclusive scan of cnt over blocks, per (h, i)
//   seg_off  1 CTA   : segment sizes from the scanned counts; exclusive scan
//                      over s -> seg_off (and, for the chunked forward, the
//                      chunk-padded output regions of the work items)
//   scatter  (blk,H) : rank of each record inside its block (per-warp bit
//                      masks + popc) + the block's base per partition (staged
//                      once per CTA) -> perm / perm_rec, and the partial-output
//                      row of every contribution (rec_pos)
#include <algorithm>

#include "sse_internal.cuh"

namespace sse {

int64_t route_max_blocks(int64_t total_tokens, int32_t num_seqs) {
    return (total_tokens + kRouteBlock - 1) / kRouteBlock + num_seqs;
}

namespace {

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of
// 32, at most 1024).  Returns the exclusive prefix; *total receives the sum.
__device__ int block_exclusive_scan(int x, int *total) {
    __shared__ int warp_off[32];
    __shared__ int s_total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();  // previous call's readers are done with warp_off / s_total
    if (lane == 31) warp_off[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? warp_off[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nwarps) warp_off[lane] = wi - w;
        if (lane == 31) s_total = wi;
    }
    __syncthreads();
    *total = s_total;
    return warp_off[warp] + incl - x;
}

// Routing blocks: each sequence is cut into blocks of kRouteBlock tokens
// (never straddling two sequences).  blk_prefix[b] = blocks before sequence b;
// blk_info[j] = (sequence, first token, end token) of block j, sequence -1 for
// the unused tail up to max_blocks.  One CTA.
__global__ void plan_blocks_kernel(const int32_t *__restrict__ cu, int32_t nseq, int32_t *__restrict__ blk_prefix,
                                   int4 *__restrict__ blk_info, int32_t max_blocks) {
    griddep_launch_dependents();
    griddep_wait();
    int carry = 0;
    for (int base = 0; base < nseq; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int nb = 0, t0 = 0, t1 = 0;
        if (b < nseq) {
            t0 = cu[b];
            t1 = cu[b + 1];
            nb = (t1 - t0 + kRouteBlock - 1) / kRouteBlock;
        }
        int tot;
        const int ex = block_exclusive_scan(nb, &tot);
        if (b < nseq) {
            blk_prefix[b] = carry + ex;
            for (int jb = 0; jb < nb; ++jb)
                blk_info[carry + ex + jb] = make_int4(b, t0 + jb * kRouteBlock, min(t0 + (jb + 1) * kRouteBlock, t1), 0);
        }
        carry += tot;
    }
    if (threadIdx.x == 0) blk_prefix[nseq] = carry;
    for (int j = carry + threadIdx.x; j < max_blocks; j += blockDim.x) blk_info[j] = make_int4(-1, 0, 0, 0);
}

template <typename T, int NP>
__global__ void __launch_bounds__(kRouteBlock)
route_count_kernel(const T *__restrict__ logits, const int4 *blk_info, int32_t H, int32_t N,
                   int32_t k, int32_t vec, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                   int32_t *__restrict__ cnt, int32_t max_blocks) {
    __shared__ int hist[kMaxPartitions];
    griddep_launch_dependents();
    if (threadIdx.x < kMaxPartitions) hist[threadIdx.x] = 0;
    griddep_wait();
    // consecutive CTAs take the heads of one routing block, so the partial
    // sectors they write into [T, H, ...] rows meet in L2
    const int h = (int)(blockIdx.x % (unsigned)H), j = (int)(blockIdx.x / (unsigned)H);
    const int4 bi = blk_info[j];  // (sequence, first token, end token); sequence -1: past the last block
    __syncthreads();
    if (bi.x >= 0) {
        const int t = bi.y + threadIdx.x;
        if (t < bi.z) {
            int idx[kMaxTopK];
            float w[kMaxTopK];
            route_token<T, NP>(logits + ((int64_t)t * H + h) * N, N, k, vec != 0, idx, w);
            const int64_t o = ((int64_t)t * H + h) * k;
            for (int jj = 0; jj < k; ++jj) {
                topk_idx[o + jj] = idx[jj];
                if (topk_w) topk_w[o + jj] = w[jj];
                atomicAdd(&hist[idx[jj]], 1);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x)
        cnt[((int64_t)h * N + i) * (max_blocks + 1) + j] = hist[i];
}

__global__ void __launch_bounds__(1024)
scan_blocks_kernel(int32_t *cnt, int32_t max_blocks) {
    griddep_launch_dependents();
    griddep_wait();
    int32_t *row = cnt + (int64_t)blockIdx.x * (max_blocks + 1);
    int carry = 0;
    for (int base = 0; base < max_blocks; base += blockDim.x) {
        const int j = base + threadIdx.x;
        const int x = j < max_blocks ? row[j] : 0;
        int tot;
        const int ex = block_exclusive_scan(x, &tot);
        if (j < max_blocks) row[j] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) row[max_blocks] = carry;
}

// Length of routed segment s = (b*H + h)*N + i from the scanned block counts.
__device__ __forceinline__ int routed_len(const int32_t *cnt, int32_t max_blocks, const int32_t *blk_prefix,
                                          int32_t H, int32_t N, int64_t s) {
    const int i = (int)(s % N);
    const int64_t bh = s / N;
    const int h = (int)(bh % H), b = (int)(bh / H);
    const int32_t *row = cnt + ((int64_t)h * N + i) * (max_blocks + 1);
    return row[blk_prefix[b + 1]] - row[blk_prefix[b]];
}

// seg_off: exclusive scan of the routed segment lengths.  pad_off (optional):
// exclusive scan over the work items (shared segments, then routed ones) of
// their lengths rounded up to whole chunks.
__global__ void __launch_bounds__(1024)
seg_off_kernel(const int32_t *cnt, int32_t max_blocks,
               const int32_t *blk_prefix, const int32_t *__restrict__ cu, int32_t nseq,
               int32_t H, int32_t N, int32_t use_shared, int32_t *__restrict__ seg_off,
               int32_t *__restrict__ pad_off) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t nseg = (int64_t)nseq * H * N;
    int carry = 0;
    for (int64_t base = 0; base < nseg; base += blockDim.x) {
        const int64_t s = base + threadIdx.x;
        const int x = s < nseg ? routed_len(cnt, max_blocks, blk_prefix, H, N, s) : 0;
        int tot;
        const int ex = block_exclusive_scan(x, &tot);
        if (s < nseg) seg_off[s] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) seg_off[nseg] = carry;
    if (!pad_off) return;
    const int64_t nshared = use_shared ? (int64_t)nseq * H : 0;
    const int64_t nitems = nshared + nseg;
    carry = 0;
    for (int64_t base = 0; base < nitems; base += blockDim.x) {
        const int64_t u = base + threadIdx.x;
        int x = 0;
        if (u < nshared) {
            const int b = (int)(u / H);
            x = cu[b + 1] - cu[b];
        } else if (u < nitems) {
            x = routed_len(cnt, max_blocks, blk_prefix, H, N, u - nshared);
        }
        x = (x + kChunkRows - 1) / kChunkRows * kChunkRows;
        int tot;
        const int ex = block_exclusive_scan(x, &tot);
        if (u < nitems) pad_off[u] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) pad_off[nitems] = carry;
}

__global__ void __launch_bounds__(kRouteBlock)
scatter_kernel(const int32_t *topk_idx, const int32_t *__restrict__ cu, int32_t nseq,
               const int32_t *blk_prefix, const int4 *blk_info,
               const int32_t *cnt, int32_t max_blocks, const int32_t *seg_off, int32_t H,
               int32_t N, int32_t k, int32_t use_shared, const float *topk_w, int32_t *__restrict__ perm,
               int32_t *__restrict__ perm_rec, float *__restrict__ perm_e,
               const int32_t *pad_off, int32_t *__restrict__ rec_pos) {
    constexpr int kWarps = kRouteBlock / 32;
    __shared__ uint32_t wmask[kWarps][kMaxPartitions];
    // per partition i: where this block's records of segment (b, h, i) start
    // in perm, and in the partial-output rows; for the shared partition, the
    // partial row of token t is s_shared + t
    __shared__ int s_base[kMaxPartitions], s_pad[kMaxPartitions], s_shared;
    // consecutive CTAs take the heads of one routing block, so the partial
    // sectors they write into [T, H, ...] rows meet in L2
    const int h = (int)(blockIdx.x % (unsigned)H), j = (int)(blockIdx.x / (unsigned)H);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    griddep_launch_dependents();
    griddep_wait();
    const int4 bi = blk_info[j];  // (sequence, first token, end token); sequence -1: past the last block
    if (bi.x < 0) return;
    const int b = bi.x;
    const int64_t nshared = use_shared ? (int64_t)nseq * H : 0;
    for (int x = threadIdx.x; x < kWarps * kMaxPartitions; x += blockDim.x)
        (&wmask[0][0])[x] = 0u;
    if (threadIdx.x < N) {
        const int i = threadIdx.x;
        const int32_t *row = cnt + ((int64_t)h * N + i) * (max_blocks + 1);
        const int before = row[j] - row[blk_prefix[b]];  // records of (b, h, i) in earlier blocks
        const int64_t seg = ((int64_t)b * H + h) * N + i;
        s_base[i] = seg_off[seg] + before;
        if (pad_off) s_pad[i] = pad_off[nshared + seg] + before;
    }
    if (threadIdx.x == kRouteBlock - 1 && rec_pos && use_shared) s_shared = pad_off[(int64_t)b * H + h] - cu[b];
    __syncthreads();
    const int t = bi.y + threadIdx.x;
    const bool valid = t < bi.z;
    int idx[kMaxTopK];
    if (valid) {
        const int64_t o = ((int64_t)t * H + h) * k;
        for (int jj = 0; jj < k; ++jj) {
            idx[jj] = topk_idx[o + jj];
            atomicOr(&wmask[warp][idx[jj]], 1u << lane);
        }
    }
    __syncthreads();
    if (!valid) return;
    const uint32_t lt = (1u << lane) - 1u;
    const int ncon = k + use_shared;
    const int64_t th = (int64_t)t * H + h;
    if (rec_pos && use_shared) rec_pos[th * ncon + k] = s_shared + t;
    for (int jj = 0; jj < k; ++jj) {
        const int i = idx[jj];
        int rank = __popc(wmask[warp][i] & lt);
        for (int w2 = 0; w2 < warp; ++w2) rank += __popc(wmask[w2][i]);
        const int64_t pos = (int64_t)s_base[i] + rank;
        if (perm) perm[pos] = t;
        if (perm_rec) perm_rec[pos] = t * k + jj;
        if (perm_e) perm_e[pos] = topk_w[th * k + jj];
        if (rec_pos) rec_pos[th * ncon + jj] = s_pad[i] + rank;
    }
}

// Router launch with the unroll bound NP >= N; rows go through 16-byte
// vector loads when every row starts on a 16-byte boundary.
template <typename T>
cudaError_t launch_count(dim3 grid, cudaStream_t stream, const T *logits, const int4 *blk_info, int32_t H, int32_t N,
                  int32_t k, int32_t *topk_idx, float *topk_w, int32_t *cnt, int32_t MB) {
    const int vec = (N * sizeof(T)) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
#define SSE_COUNT(NP)                                                                                         \
    launch_dependent(route_count_kernel<T, NP>, grid, dim3(kRouteBlock), 0, stream, logits, blk_info, H, N, k, vec, \
                     topk_idx, topk_w, cnt, MB)
    if (N <= 8) return SSE_COUNT(8);
    if (N <= 16) return SSE_COUNT(16);
    if (N <= 32) return SSE_COUNT(32);
    return SSE_COUNT(64);
#undef SSE_COUNT
}

// Masking schedule: item u's output rows start at pad_off[u].  With pl_b the
// length of sequence b rounded up to whole chunks and P_b their exclusive
// prefix: shared item (b, h) -> H P_b + h pl_b; item (b, h, i) -> (shared
// total) + H N P_b + (h N + i) pl_b.  One CTA.
__global__ void __launch_bounds__(1024)
masked_pad_kernel(const int32_t *__restrict__ cu, int32_t nseq, int32_t H, int32_t N, int32_t use_shared,
                  int32_t *__restrict__ pad_off) {
    extern __shared__ int s_pref[];  // [nseq + 1]
    griddep_launch_dependents();
    griddep_wait();
    int carry = 0;
    for (int base = 0; base < nseq; base += blockDim.x) {
        const int b = base + threadIdx.x;
        const int pl = b < nseq ? (cu[b + 1] - cu[b] + kChunkRows - 1) / kChunkRows * kChunkRows : 0;
        int tot;
        const int ex = block_exclusive_scan(pl, &tot);
        if (b < nseq) s_pref[b] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) s_pref[nseq] = carry;
    __syncthreads();
    const int64_t nshared = use_shared ? (int64_t)nseq * H : 0;
    const int64_t shared_rows = use_shared ? (int64_t)H * s_pref[nseq] : 0;
    const int64_t nitems = nshared + (int64_t)nseq * H * N;
    for (int64_t u = threadIdx.x; u < nitems; u += blockDim.x) {
        int64_t v;
        if (u < nshared) {
            const int b = (int)(u / H), h = (int)(u % H);
            const int pl = s_pref[b + 1] - s_pref[b];
            v = (int64_t)H * s_pref[b] + (int64_t)h * pl;
        } else {
            const int64_t r = u - nshared;
            const int b = (int)(r / ((int64_t)H * N));
            const int hi = (int)(r % ((int64_t)H * N));  // h * N + i
            const int pl = s_pref[b + 1] - s_pref[b];
            v = shared_rows + (int64_t)H * N * s_pref[b] + (int64_t)hi * pl;
        }
        pad_off[u] = (int32_t)v;
    }
    if (threadIdx.x == 0) pad_off[nitems] = (int32_t)(shared_rows + (int64_t)H * N * s_pref[nseq]);
}

// Partial row of each contribution of (t, h): selected partition j of the
// token, then the shared one.
__global__ void __launch_bounds__(256)
masked_recpos_kernel(const int32_t *__restrict__ cu, int32_t nseq, const int32_t *topk_idx,
                     int64_t total_tokens, int32_t H, int32_t N, int32_t k, int32_t use_shared,
                     const int32_t *pad_off, int32_t *__restrict__ rec_pos) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t rows = total_tokens * H;
    const int ncon = k + use_shared;
    const int64_t nshared = use_shared ? (int64_t)nseq * H : 0;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < rows; x += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(x / H), h = (int)(x % H);
        int lo = 0, hi = nseq - 1;  // the sequence holding t: largest b with cu[b] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int b = lo, dt = t - cu[b];
        for (int j = 0; j < k; ++j) {
            const int i = topk_idx[x * k + j];
            rec_pos[x * ncon + j] = pad_off[nshared + ((int64_t)b * H + h) * N + i] + dt;
        }
        if (use_shared) rec_pos[x * ncon + k] = pad_off[(int64_t)b * H + h] + dt;
    }
}

}  // namespace

cudaError_t launch_route(const sse_config_t &cfg, const void *logits, const int32_t *cu_seqlens,
                         int32_t num_seqs, int64_t total_tokens, const RouteBuffers &rb,
                         bool group, cudaStream_t stream) {
    const int H = cfg.num_heads, N = cfg.num_partitions, k = cfg.top_k;
    const int MB = rb.max_blocks;
    plan_blocks_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, num_seqs, rb.blk_prefix, rb.blk_info, MB);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((int64_t)MB * H));
    e = cfg.dtype == SSE_BF16
            ? launch_count<__nv_bfloat16>(grid, stream, static_cast<const __nv_bfloat16 *>(logits), rb.blk_info, H, N,
                                          k, rb.topk_idx, rb.topk_w, rb.cnt, MB)
            : launch_count<float>(grid, stream, static_cast<const float *>(logits), rb.blk_info, H, N, k,
                                  rb.topk_idx, rb.topk_w, rb.cnt, MB);
    if (e != cudaSuccess || !group) return e;
    e = launch_dependent(scan_blocks_kernel, dim3(H * N), dim3(1024), 0, stream, rb.cnt, MB);
    if (e != cudaSuccess) return e;
    e = launch_dependent(seg_off_kernel, dim3(1), dim3(1024), 0, stream, (const int32_t *)rb.cnt, MB,
                         (const int32_t *)rb.blk_prefix, cu_seqlens, num_seqs, H, N, cfg.use_shared, rb.seg_off,
                         rb.pad_off);
    if (e != cudaSuccess) return e;
    return launch_dependent(scatter_kernel, grid, dim3(kRouteBlock), 0, stream, (const int32_t *)rb.topk_idx,
                            cu_seqlens, num_seqs, (const int32_t *)rb.blk_prefix, (const int4 *)rb.blk_info,
                            (const int32_t *)rb.cnt, MB, (const int32_t *)rb.seg_off, H, N, k, cfg.use_shared,
                            (const float *)rb.topk_w, rb.perm, rb.perm_rec, rb.perm_e, (const int32_t *)rb.pad_off,
                            rb.rec_pos);
}

}  // namespace sse

namespace sse {

cudaError_t launch_masked_plan(const sse_config_t &cfg, const int32_t *cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, const RouteBuffers &rb, cudaStream_t stream) {
    masked_pad_kernel<<<1, 1024, sizeof(int) * (num_seqs + 1), stream>>>(cu_seqlens, num_seqs, cfg.num_heads,
                                                                         cfg.num_partitions, cfg.use_shared,
                                                                         rb.pad_off);
    const int64_t rows = total_tokens * cfg.num_heads;
    if (rows > 0) {
        const unsigned blocks = (unsigned)std::min<int64_t>((rows + 255) / 256, 152 * 8);
        masked_recpos_kernel<<<blocks, 256, 0, stream>>>(cu_seqlens, num_seqs, rb.topk_idx, total_tokens,
                                                        cfg.num_heads, cfg.num_partitions, cfg.top_k,
                                                        cfg.use_shared, rb.pad_off, rb.rec_pos);
    }
    return cudaGetLastError();
}

}  // namespace sse
