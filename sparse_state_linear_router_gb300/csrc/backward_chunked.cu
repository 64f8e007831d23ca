// backward_chunked.cu -- gradients of the SSE layer ("Scaling Linear Attention
// with Sparse State Expansion", eqs. 9-14, the shared partition of section 2.5
// and the varlen schedule of section 2.6) in chunked form on the tensor cores,
// for key dimension c = 128 and bf16 tokens.
//
// Notation of one work item (a routed segment (b, h, i) in time order, or the
// shared partition of (b, h) over the whole sequence), as in backward.cu:
//   Q_t = w_t q_t with w = e_t scale (routed) or scale (shared); K_t = e_t k_t;
//   S_t = diag(a_t) S_{t-1} + K_t^T v_t;  o_t gets Q_t S_t.
// The item's rows are cut into chunks of 128.  In a chunk with rows
// r = 0..127, G_r is the running sum of g from the chunk's first row through
// row r, G_m its value at the midpoint row (63) and G_l at the last row.
//
//   forward state contributions:  U_j = K_hat^T V, K_hat_r = exp(G_l - G_r) K_r
//   backward ones:                W_j = Q_hat^T dO, Q_hat_r = exp(G_r) Q_r
//   scan over chunks (elementwise over c x d):
//     S_start[j + 1] = diag(exp(G_l,j)) S_start[j] + U_j          S_start[0] = S_0
//     dS_end[j - 1]  = diag(exp(G_l,j)) dS_end[j] + W_j           dS_end[last] = dL/dS_T
//   and dL/dS_0 = diag(exp(G_l,0)) dS_end[0] + W_0.
//
// Inside chunk j, with Qt_r = Q_r exp(G_r - G_m), Kt_r = K_r exp(G_m - G_r),
// S' = diag(exp(G_m)) S_start[j], dS' = diag(exp(G_l - G_m)) dS_end[j] and
// the lower-triangular masks (row >= column) of A = Qt Kt^T and P = dO V^T:
//   U  = tril(P) Kt + dO S'^T            u_r  = exp(G_r - G_m) * U_r = S_r do_r^T
//   DK = tril(P)^T Qt + V dS'^T          dK_r = exp(G_m - G_r) * DK_r = dS_r v_r^T
//   DV = tril(A)^T dO + Kt dS'           dV_r = DV_r = K_r dS_r
// -- eight 128 x 128 x 128 products per chunk, as the per-token recurrence of
// backward.cu gives them row by row.  Then dq = w u, de(read) = scale q . u,
// dk = e dK, de(write) = k . dK, dv = dV, and the gate gradient is the reverse
// running sum over the item's rows of q * dq - k * dk, started at
// rowsum(S_T * dL/dS_T).  Every factor exp(+-(G_r - G_m)) stays within e^64
// when both |G_m| and |G_l - G_m| do; an item with a chunk past that range is
// queued for the per-token kernel, which recomputes all of its slots.
//
// Kernels (one stream, in order): chunk sums (tensor cores) -> scan (CUDA
// cores, in place) -> chunk gradients (tensor cores; they also leave each
// chunk's gate-gradient column totals) -> the reverse running sums (each
// chunk starting from the totals of its item's later chunks) -> the per-token
// kernel on the queued items -> the per-token combine of backward.cu.  The dq, dk and dv slots are bf16 (each
// value is one product, rounded once); the gate-gradient slots stay float32,
// since the running sums accumulate in place.
#include <algorithm>

#include "chunk_tiles.cuh"
#include "sse_internal.cuh"
#include "umma.cuh"

namespace sse {
namespace {

using namespace umma;
using namespace tiles;

constexpr int kRows = kChunkRows;  // 128 rows per chunk
constexpr int kKey = 128;          // c
constexpr int kThr = 256;          // 8 warps: two per TMEM lane quarter
constexpr uint32_t kTile = 128 * 256;
static_assert(kThr - kRows == kKey, "the upper half of the CTA writes one chunk total per column");
constexpr float kRange = 64.f;     // largest |G_m| and |G_l - G_m| the factorised form takes
#ifdef SSE_FAULT_INJECT
// Checked build (libsse_checked.so, for the failure-detection test only):
// every bounded wait gives up after 50 ms, and g_bwd_fault_mode = 1 makes
// CTA 0 of the gradient kernel issue neither the first product round of its
// first chunk nor its commit, so that the wait on it runs out and the kernel
// takes its abort path (SSE_DEVICE_TIMEOUT, TMEM freed) with no product in
// flight.
__device__ int g_bwd_fault_mode = 0;
constexpr uint64_t kWait = 50000000ull;
#else
constexpr uint64_t kWait = 2000000000ull;
#endif

// The work item and chunk of global chunk index `chunk` (items own the
// chunk-padded row ranges pad_off[u] .. pad_off[u + 1]).  Returns false past
// the last chunk.
struct ChunkRef {
    int item, n;         // work item, chunk index inside it
    int b, h, slot;      // sequence, head, partition (N: shared)
    int base, len;       // first row (token or grouped record) and rows of the item
    bool shared;
};
__device__ bool locate_chunk(const BackwardArgs &a, int64_t chunk, int H, int N, int use_shared, ChunkRef &r) {
    const int nshared = use_shared ? a.num_seqs * H : 0;
    const int nitems = nshared + a.num_seqs * H * N;
    const int64_t row = chunk * kRows;
    if (nitems == 0 || row >= a.pad_off[nitems]) return false;
    int lo = 0, hi = nitems - 1;  // last item with pad_off[item] <= row
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.pad_off[mid] <= row) lo = mid; else hi = mid - 1;
    }
    r.item = lo;
    r.n = (int)((row - a.pad_off[lo]) / kRows);
    r.shared = lo < nshared;
    if (r.shared) {
        r.b = lo / H;
        r.h = lo % H;
        r.slot = N;
        r.base = a.cu_seqlens[r.b];
        r.len = a.cu_seqlens[r.b + 1] - r.base;
    } else {
        const int s = lo - nshared;
        r.slot = s % N;
        r.h = (s / N) % H;
        r.b = s / (N * H);
        r.base = a.seg_off[s];
        r.len = a.seg_off[s + 1] - r.base;
    }
    return true;
}

// Row metadata of row x (< 128) of a chunk: token, router weight, slot j of
// the token's contributions (its top-k place, k for the shared partition);
// token -1 past the item's end.
__device__ __forceinline__ void row_meta(const BackwardArgs &a, const ChunkRef &r, int x, int topk, int &t, float &e,
                                         int &j) {
    const int idx = r.n * kRows + x;
    t = -1;
    e = 0.f;
    j = 0;
    if (idx >= r.len) return;
    if (r.shared) {
        t = r.base + idx;
        e = 1.f;
        j = topk;
    } else {
        const int rec = a.perm_rec[r.base + idx];
        t = rec / topk;
        j = rec - t * topk;
        e = a.perm_e[r.base + idx];
    }
}

// Per-column gate sums of a staged g tile: thread (col, half) sums rows
// half * 64 .. half * 64 + 63 of column col into part[half][col].
__device__ __forceinline__ void gate_half_sums(const unsigned char *tg, float *part) {
    const int col = threadIdx.x & (kKey - 1), half = threadIdx.x >> 7;
    float s = 0.f;
#pragma unroll 8
    for (int x = half * 64; x < half * 64 + 64; ++x)
        s += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tg + toff(x, col)));
    part[half * kKey + col] = s;
}

// Shared memory of the chunk kernels: tiles from a 1024-aligned base, then
// row metadata, gate sums, the mbarrier and the TMEM address slot.
struct ChunkSmem {
    unsigned char *tile[6];
    int *tok, *slotj;
    float *e, *part, *gm, *gl, *de, *patch, *csum;
    uint32_t bar;
    uint32_t *tslot;
};
__device__ __forceinline__ ChunkSmem carve_smem(unsigned char *raw, int ntiles) {
    unsigned char *sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    ChunkSmem c;
    for (int i = 0; i < 6; ++i) c.tile[i] = sm + (i < ntiles ? i : 0) * kTile;
    unsigned char *p = sm + ntiles * kTile;
    c.tok = reinterpret_cast<int *>(p);   // [2 buffers][kRows]
    c.slotj = c.tok + 2 * kRows;          // [2][kRows]
    c.e = reinterpret_cast<float *>(c.slotj + 2 * kRows);  // [2][kRows]
    c.part = c.e + 2 * kRows;   // [2][kKey]
    c.gm = c.part + 2 * kKey;   // [kKey]
    c.gl = c.gm + kKey;         // [kKey]
    c.de = c.gl + kKey;         // [2 halves][2 (read, write)][kRows]
    c.patch = c.de + 4 * kRows; // [8 warps][32][kPatchStride]
    c.csum = c.patch + 8 * 32 * kPatchStride;  // [4 lane quarters][kKey]
    uint64_t *b = reinterpret_cast<uint64_t *>(c.csum + 4 * kKey);
    c.bar = smem_u32(b);
    c.tslot = reinterpret_cast<uint32_t *>(b + 1);
    return c;
}
constexpr size_t chunk_smem_bytes(int ntiles) {
    return 1024 + (size_t)ntiles * kTile + 6 * kRows * 4 + 4 * kKey * 4 + 4 * kRows * 4 +
           8 * 32 * kPatchStride * 4 + 4 * kKey * 4 + 16;
}

// Row metadata of the chunk into metadata buffer mb (threads 0..127).
__device__ __forceinline__ void chunk_meta(const BackwardArgs &a, const ChunkRef &r, int topk, const ChunkSmem &c,
                                           int mb) {
    if (threadIdx.x < kRows) {
        int t, j;
        float e;
        row_meta(a, r, threadIdx.x, topk, t, e, j);
        c.tok[mb * kRows + threadIdx.x] = t;
        c.e[mb * kRows + threadIdx.x] = e;
        c.slotj[mb * kRows + threadIdx.x] = j;
    }
}

// One elected thread issues the products through `issue` (unless `withhold`:
// the checked build's fault switch), commits them to the CTA's mbarrier and
// every thread waits (bounded).  Shared-memory operands written by the
// generic proxy before the call are made visible to the tensor core first.
// Returns false, in every thread, when the wait ran out.
template <typename F>
__device__ __forceinline__ bool run_mma(const ChunkSmem &c, uint32_t &phase, F issue, bool withhold = false) {
    fence_proxy_async();
    fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && !withhold) {
        fence_after();
        issue();
        commit(c.bar);
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(c.bar, phase, kWait);
    phase ^= 1u;
    fence_after();
    return __syncthreads_and(ok) != 0;
}

// ---- chunk sums ---------------------------------------------------------
// U_j = K_hat^T V and W_j = Q_hat^T dO of every chunk (bf16, [c][d] each) and
// gamma_j = exp(G_l).  Persistent CTAs walk the chunks; per chunk: stage the
// raw q, k, g, v, dO rows; per-column gate sums in two halves; K_hat, Q_hat in
// place; two products (M = c, K = the chunk's rows, N = d) into TMEM; read-out.
template <int DV>
__global__ void __launch_bounds__(kThr, 1)
bwd_chunk_sums_kernel(BackwardArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared, float scale) {
    extern __shared__ unsigned char smem_raw[];
    const ChunkSmem c = carve_smem(smem_raw, 5);
    unsigned char *tK = c.tile[0], *tV = c.tile[1], *tQ = c.tile[2], *tD = c.tile[3], *tG = c.tile[4];
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) tmem_alloc(smem_u32(c.tslot), 256);
    if (tid == 0) {
        mbar_init(c.bar, 1);
        mbar_fence_init();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *c.tslot;
    uint32_t phase = 0;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q), *k = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *qs = static_cast<const __nv_bfloat16 *>(a.qs), *ks = static_cast<const __nv_bfloat16 *>(a.ks);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v), *g = static_cast<const __nv_bfloat16 *>(a.g);
    const __nv_bfloat16 *dout = static_cast<const __nv_bfloat16 *>(a.d_out);
    bool failed = false;
    // metadata and row staging of chunk n + 1 are issued before chunk n's read-out
    auto stage = [&](const ChunkRef &r, int mb) {
        chunk_meta(a, r, topk, c, mb);
        __syncthreads();
        const int *tok = c.tok + mb * kRows;
        stage_rows_n<kKey, 3>({tK, tQ, tG}, {r.shared && ks ? ks : k, r.shared && qs ? qs : q, g}, tok, H, r.h);
        stage_rows_n<DV, 2>({tV, tD}, {v, dout}, tok, H, r.h);
    };
    int64_t chunk = blockIdx.x;
    ChunkRef r;
    bool have = chunk < a.num_chunks && locate_chunk(a, chunk, H, N, use_shared, r);
    int mb = 0;
    if (have) stage(r, 0);
    while (have) {
        const float *ev = c.e + mb * kRows;
        cp_async_wait_all();
        __syncthreads();
        gate_half_sums(tG, c.part);
        __syncthreads();
        {
            // thread (col, half): rows half * 64 .. + 63, running G from the chunk's start
            const int col = tid & (kKey - 1), half = tid >> 7;
            const float gl = c.part[col] + c.part[kKey + col];
            float run = half ? c.part[col] : 0.f;
            if (half == 0) {
                a.gamma[chunk * kKey + col] = expf(gl);
                a.gml[chunk * 2 * kKey + col] = c.part[col];  // G_m: through the midpoint row
                a.gml[chunk * 2 * kKey + kKey + col] = gl;
            }
            for (int x = half * 64; x < half * 64 + 64; ++x) {
                run += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tG + toff(x, col)));
                const float e = ev[x];
                __nv_bfloat16 *pk = reinterpret_cast<__nv_bfloat16 *>(tK + toff(x, col));
                __nv_bfloat16 *pq = reinterpret_cast<__nv_bfloat16 *>(tQ + toff(x, col));
                // factors rounded to bf16 with the products: fast exponentials suffice
                *pk = __float2bfloat16_rn(e * __bfloat162float(*pk) * __expf(gl - run));
                *pq = __float2bfloat16_rn(e * scale * __bfloat162float(*pq) * __expf(run));
            }
        }
        const bool ok = run_mma(c, phase, [&] {
            constexpr uint32_t id = idesc_bf16(128, DV, 1, 1);  // A = tile^T (MN-major), B MN-major
            for (int k16 = 0; k16 < kRows; k16 += 16) {
                const uint32_t ro = (k16 / 8) * 2048;
                mma_bf16(tmem, desc_sw128(smem_u32(tK) + ro, 1024, 2048), desc_sw128(smem_u32(tV) + ro, 1024, 2048),
                         id, k16 > 0);
                mma_bf16(tmem + 128, desc_sw128(smem_u32(tQ) + ro, 1024, 2048),
                         desc_sw128(smem_u32(tD) + ro, 1024, 2048), id, k16 > 0);
            }
        });
        if (!ok) {
            failed = true;
            break;
        }
        const int64_t next = chunk + gridDim.x;
        ChunkRef rn;
        const bool have_next = next < a.num_chunks && locate_chunk(a, next, H, N, use_shared, rn);
        if (have_next) stage(rn, mb ^ 1);
        {
            // lane quarter (warp % 4) holds state rows 32 (warp % 4) .. + 31, column half warp / 4
            const int lane = tid & 31, hc = warp >> 2;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            float *patch = c.patch + warp * 32 * kPatchStride;
            int64_t sr[4];  // rows this lane stores: state rows of the chunk
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) sr[kk] = chunk * kKey + 32 * (warp & 3) + (lane >> 2) + 8 * kk;
            for (int c0 = hc * (DV / 2); c0 < (hc + 1) * (DV / 2); c0 += 32) {
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    uint32_t x[32], w[16];
                    tmem_ld32(tmem + lb + 128 * m + c0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
                    warp_put32_bf16(patch, lane, w, m ? a.wgrad : a.ustate, DV, c0, sr);
                }
            }
        }
        fence_before();
        __syncthreads();  // TMEM is reused by the next chunk
        chunk = next;
        r = rn;
        have = have_next;
        mb ^= 1;
    }
    if (failed) cp_async_wait_all();  // no copy may still be writing shared memory when the CTA exits
    if (failed && tid == 0) atomicOr(a.flags, SSE_DEVICE_TIMEOUT);
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// (b, h, slot) of work item u: shared (b, h) first, then routed (b, h, i).
__device__ __forceinline__ void item_bhs(int u, int H, int N, int nshared, int &b, int &h, int &slot) {
    if (u < nshared) {
        b = u / H;
        h = u % H;
        slot = N;
    } else {
        const int s = u - nshared;
        slot = s % N;
        h = (s / N) % H;
        b = s / (N * H);
    }
}

// ---- scan over chunks ---------------------------------------------------------
// One thread per four elements of an item's c x d state: forward, the state
// at chunk j's start, S' = diag(exp(G_m)) S_start; backward, dL/dS at its end,
// dS' = diag(exp(G_l - G_m)) dS_end -- each written in bf16 straight into the
// operand tile layout the gradient kernel copies in.  Also
// rowsum(S_T * dL/dS_T) into fterm and dL/dS_0 into d_init.
template <int DV>
__global__ void __launch_bounds__(256)
bwd_state_scan_kernel(BackwardArgs a, int32_t H, int32_t N, int32_t use_shared) {
    constexpr int Q4 = DV / 4;  // float4 per state row: one warp (d = 128) or half of one (d = 64)
    const int u = blockIdx.x;
    const int nshared = use_shared ? a.num_seqs * H : 0;
    int b, h, slot;
    item_bhs(u, H, N, nshared, b, h, slot);
    const int P = N + use_shared;
    const int e4 = blockIdx.y * blockDim.x + threadIdx.x;
    const int row = e4 / Q4, col = (e4 % Q4) * 4;
    const int64_t cb = a.pad_off[u] / kRows;
    const int nch = (a.pad_off[u + 1] - a.pad_off[u]) / kRows;
    const int64_t so = (((int64_t)b * H + h) * P + slot) * (int64_t)kKey * DV + (int64_t)row * DV + col;
    const int64_t cs = (int64_t)kKey * DV / 4;  // stride between chunks, in four-element pieces
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint2 *U = reinterpret_cast<const uint2 *>(a.ustate + (cb * kKey + row) * DV + col);
    const uint2 *W = reinterpret_cast<const uint2 *>(a.wgrad + (cb * kKey + row) * DV + col);
    auto f4 = [](uint2 u) {
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    };
    const float *gam = a.gamma + cb * kKey + row;
    const float *gml = a.gml + cb * 2 * kKey + row;  // G_m at [j][0][row], G_l at [j][1][row]
    const uint32_t toffs = toff(row, col);           // four bf16 in one 8-byte piece
    unsigned char *sp = static_cast<unsigned char *>(a.sp_tiles) + cb * (int64_t)kTile + toffs;
    unsigned char *dsp = static_cast<unsigned char *>(a.dsp_tiles) + cb * (int64_t)kTile + toffs;
    auto put4 = [](unsigned char *p, float f, float4 x) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(pack2(f * x.x, f * x.y), pack2(f * x.z, f * x.w));
    };

    // eight chunks' loads in flight ahead of the dependent updates
    constexpr int kAhead = 8;
    float4 S = a.init ? *reinterpret_cast<const float4 *>(a.init + so) : zero;
    for (int j0 = 0; j0 < nch; j0 += kAhead) {
        float4 x[kAhead];
        float gm[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
            x[i] = j0 + i < nch ? f4(U[(j0 + i) * cs]) : zero;
            gm[i] = j0 + i < nch ? gam[(int64_t)(j0 + i) * kKey] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
            if (j0 + i >= nch) break;
            put4(sp + (int64_t)(j0 + i) * kTile, expf(gml[(int64_t)(j0 + i) * 2 * kKey]), S);
            S = make_float4(fmaf(gm[i], S.x, x[i].x), fmaf(gm[i], S.y, x[i].y), fmaf(gm[i], S.z, x[i].z),
                            fmaf(gm[i], S.w, x[i].w));
        }
    }
    const float4 df = a.d_final ? *reinterpret_cast<const float4 *>(a.d_final + so) : zero;
    float pr = S.x * df.x + S.y * df.y + S.z * df.z + S.w * df.w;
#pragma unroll
    for (int o = Q4 / 2; o > 0; o >>= 1) pr += __shfl_xor_sync(0xffffffffu, pr, o);
    if (threadIdx.x % Q4 == 0) a.fterm[(int64_t)u * kKey + row] = pr;

    float4 dS = df;
    for (int j0 = nch - 1; j0 >= 0; j0 -= kAhead) {
        float4 x[kAhead];
        float gm[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
            x[i] = j0 - i >= 0 ? f4(W[(j0 - i) * cs]) : zero;
            gm[i] = j0 - i >= 0 ? gam[(int64_t)(j0 - i) * kKey] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
            if (j0 - i < 0) break;
            const float *gj = gml + (int64_t)(j0 - i) * 2 * kKey;
            put4(dsp + (int64_t)(j0 - i) * kTile, expf(gj[kKey] - gj[0]), dS);
            dS = make_float4(fmaf(gm[i], dS.x, x[i].x), fmaf(gm[i], dS.y, x[i].y), fmaf(gm[i], dS.z, x[i].z),
                             fmaf(gm[i], dS.w, x[i].w));
        }
    }
    if (a.d_init) *reinterpret_cast<float4 *>(a.d_init + so) = dS;
}

// bf16 x 8 of a 16-byte global load
__device__ __forceinline__ void unpack8(uint4 w, float (&f)[8]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(ws[i] << 16);
        f[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
    }
}

// ---- chunk gradients --------------------------------------------------------
// Per chunk, with six 32 KB tiles: Qt (tile 0), Kt (1), V (2), dO (3), tile 4
// (the raw g rows, then tril(A), then dS'), tile 5 (tril(P)); tile 0 takes S'
// once the products that read Qt are done.  TMEM columns: [0, 128) A then U,
// [128, 256) P then DK, [256, 256 + d) DV.
template <int DV>
__global__ void __launch_bounds__(kThr, 1)
bwd_chunk_grads_kernel(BackwardArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared, float scale) {
    extern __shared__ unsigned char smem_raw[];
    const ChunkSmem c = carve_smem(smem_raw, 6);
    unsigned char *tQ = c.tile[0], *tK = c.tile[1], *tV = c.tile[2], *tD = c.tile[3], *tA = c.tile[4],
                  *tP = c.tile[5];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) tmem_alloc(smem_u32(c.tslot), 512);
    if (tid == 0) {
        mbar_init(c.bar, 1);
        mbar_fence_init();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *c.tslot;
    uint32_t phase = 0;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q), *k = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *qs = static_cast<const __nv_bfloat16 *>(a.qs), *ks = static_cast<const __nv_bfloat16 *>(a.ks);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v), *g = static_cast<const __nv_bfloat16 *>(a.g);
    const __nv_bfloat16 *dout = static_cast<const __nv_bfloat16 *>(a.d_out);
    float *gs = a.gscratch + (int64_t)blockIdx.x * kRows * kKey;  // G_r - G_m of the chunk in flight
    const int ncon = topk + use_shared;
    // epilogue / mask layout: lane quarter (warp % 4) = rows, column half = warp / 4
    const int quarter = warp & 3, hc = warp >> 2, erow = 32 * quarter + lane;
    const uint32_t lb = (uint32_t)(32 * quarter) << 16;
    bool failed = false;
#ifdef SSE_FAULT_INJECT
    bool first_chunk = true;  // of this CTA (the checked build's fault switch)
#endif
    // metadata and row staging of chunk n + 1 are issued once chunk n's last
    // products are done (every tile free), before its read-out
    auto stage = [&](const ChunkRef &r, int mb) {
        chunk_meta(a, r, topk, c, mb);
        __syncthreads();
        const int *tok = c.tok + mb * kRows;
        stage_rows_n<kKey, 3>({tQ, tK, tA}, {r.shared && qs ? qs : q, r.shared && ks ? ks : k, g}, tok, H, r.h);
        stage_rows_n<DV, 2>({tV, tD}, {v, dout}, tok, H, r.h);
    };
    int64_t chunk = blockIdx.x;
    ChunkRef r;
    bool have = chunk < a.num_chunks && locate_chunk(a, chunk, H, N, use_shared, r);
    int mb = 0;
    if (have) stage(r, 0);
    while (have) {
        const int *tok = c.tok + mb * kRows, *sj = c.slotj + mb * kRows;
        const float *ev = c.e + mb * kRows;
        cp_async_wait_all();
        __syncthreads();
        gate_half_sums(tA, c.part);
        __syncthreads();
        bool bad;
        {
            // thread (col, half): rows half * 64 .. + 63; G_m closes the first half
            const int col = tid & (kKey - 1), half = tid >> 7;
            const float gm = c.part[col], gl = gm + c.part[kKey + col];
            bad = fabsf(gm) > kRange || fabsf(gl - gm) > kRange;
            if (half == 0) {
                c.gm[col] = gm;
                c.gl[col] = gl;
            }
            float run = half ? gm : 0.f;
            for (int x = half * 64; x < half * 64 + 64; ++x) {
                run += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tA + toff(x, col)));
                const float d = run - gm, e = ev[x];
                __nv_bfloat16 *pq = reinterpret_cast<__nv_bfloat16 *>(tQ + toff(x, col));
                __nv_bfloat16 *pk = reinterpret_cast<__nv_bfloat16 *>(tK + toff(x, col));
                *pq = __float2bfloat16_rn(e * scale * __bfloat162float(*pq) * __expf(d));
                *pk = __float2bfloat16_rn(e * __bfloat162float(*pk) * __expf(-d));
                gs[x * kKey + col] = d;
            }
        }
        // a chunk past the gate range: the item is queued once for the per-token kernel
        if (__syncthreads_or(bad) && tid == 0 && atomicExch(a.marks + r.item, 1) == 0) {
            atomicOr(a.flags, SSE_DEVICE_RECOMPUTED);
            a.redo_list[atomicAdd(a.flags + 1, 1)] = r.item;
        }
        // products 1: A = Qt Kt^T, P = dO V^T
#ifdef SSE_FAULT_INJECT
        const bool withhold = g_bwd_fault_mode == 1 && blockIdx.x == 0 && first_chunk;
        first_chunk = false;
#else
        const bool withhold = false;
#endif
        bool ok = run_mma(c, phase, [&] {
            constexpr uint32_t id = idesc_bf16(128, 128, 0, 0);
            for (int k16 = 0; k16 < kKey; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                mma_bf16(tmem, desc_sw128(smem_u32(tQ) + ko, 16, 2048), desc_sw128(smem_u32(tK) + ko, 16, 2048), id,
                         k16 > 0);
            }
            for (int k16 = 0; k16 < DV; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                mma_bf16(tmem + 128, desc_sw128(smem_u32(tD) + ko, 16, 2048), desc_sw128(smem_u32(tV) + ko, 16, 2048),
                         id, k16 > 0);
            }
        }, withhold);
        if (!ok) {
            failed = true;
            break;
        }
        // tril(A) -> tile 4, tril(P) -> tile 5 (bf16)
        for (int c0 = hc * 64; c0 < hc * 64 + 64; c0 += 32) {
            uint32_t x[32];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                tmem_ld32(tmem + lb + 128 * m + c0, x);
                tmem_wait_ld();
                unsigned char *dst = m ? tP : tA;
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    float f[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) f[jj] = c0 + i + jj <= erow ? __uint_as_float(x[i + jj]) : 0.f;
                    *reinterpret_cast<uint4 *>(dst + toff(erow, c0 + i)) =
                        make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
                }
            }
        }
        // products 2: U = tril(P) Kt, DK = tril(P)^T Qt, DV = tril(A)^T dO
        ok = run_mma(c, phase, [&] {
            constexpr uint32_t idU = idesc_bf16(128, 128, 0, 1), idK = idesc_bf16(128, 128, 1, 1);
            constexpr uint32_t idV = idesc_bf16(128, DV, 1, 1);
            for (int k16 = 0; k16 < kRows; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2, ro = (k16 / 8) * 2048;
                mma_bf16(tmem, desc_sw128(smem_u32(tP) + ko, 16, 2048), desc_sw128(smem_u32(tK) + ro, 1024, 2048), idU,
                         k16 > 0);
                mma_bf16(tmem + 128, desc_sw128(smem_u32(tP) + ro, 1024, 2048),
                         desc_sw128(smem_u32(tQ) + ro, 1024, 2048), idK, k16 > 0);
                mma_bf16(tmem + 256, desc_sw128(smem_u32(tA) + ro, 1024, 2048),
                         desc_sw128(smem_u32(tD) + ro, 1024, 2048), idV, k16 > 0);
            }
        });
        if (!ok) {
            failed = true;
            break;
        }
        // S' -> tile 0 and dS' -> tile 4: the scan wrote them in the tile layout
        {
            const unsigned char *sp = static_cast<const unsigned char *>(a.sp_tiles) + chunk * (int64_t)kTile;
            const unsigned char *dsp = static_cast<const unsigned char *>(a.dsp_tiles) + chunk * (int64_t)kTile;
            for (int x = tid; x < (int)(kTile / 16); x += kThr) {
                cp_async16(smem_u32(tQ + 16 * x), sp + 16 * x, true);
                cp_async16(smem_u32(tA + 16 * x), dsp + 16 * x, true);
            }
            cp_async_wait_all();
        }
        // products 3: U += dO S'^T, DK += V dS'^T, DV += Kt dS'
        ok = run_mma(c, phase, [&] {
            constexpr uint32_t idT = idesc_bf16(128, 128, 0, 0), idV = idesc_bf16(128, DV, 0, 1);
            for (int k16 = 0; k16 < DV; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                mma_bf16(tmem, desc_sw128(smem_u32(tD) + ko, 16, 2048), desc_sw128(smem_u32(tQ) + ko, 16, 2048), idT, 1);
                mma_bf16(tmem + 128, desc_sw128(smem_u32(tV) + ko, 16, 2048), desc_sw128(smem_u32(tA) + ko, 16, 2048),
                         idT, 1);
            }
            for (int k16 = 0; k16 < kKey; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2, ro = (k16 / 8) * 2048;
                mma_bf16(tmem + 256, desc_sw128(smem_u32(tK) + ko, 16, 2048),
                         desc_sw128(smem_u32(tA) + ro, 1024, 2048), idV, 1);
            }
        });
        if (!ok) {
            failed = true;
            break;
        }
        const int64_t next = chunk + gridDim.x;
        ChunkRef rn;
        const bool have_next = next < a.num_chunks && locate_chunk(a, next, H, N, use_shared, rn);
        if (have_next) stage(rn, mb ^ 1);
        // read-out: row erow of U, DK (columns of this warp's half) and DV; the
        // slot rows of a warp's 32 rows are scattered, so every value goes out
        // through the warp's store patch
        {
            const int t = tok[erow];
            const float e = ev[erow];
            const bool valid = t >= 0;
            const int64_t th = (int64_t)(valid ? t : 0) * H + r.h;
            const __nv_bfloat16 *qrow = (r.shared && qs ? qs : q) + th * kKey;
            const __nv_bfloat16 *krow = (r.shared && ks ? ks : k) + th * kKey;
            const float *gsr = gs + erow * kKey;
            float *patch = c.patch + warp * 32 * kPatchStride;
            __nv_bfloat16 *dq_c = static_cast<__nv_bfloat16 *>(a.dq_c), *dk_c = static_cast<__nv_bfloat16 *>(a.dk_c);
            __nv_bfloat16 *dv_c = static_cast<__nv_bfloat16 *>(a.dv_c);
            int64_t sr[4];  // slot rows this lane stores (-1 past the item's end)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int rr = 32 * quarter + (lane >> 2) + 8 * kk, tt = tok[rr];
                sr[kk] = tt >= 0 ? ((int64_t)tt * H + r.h) * ncon + sj[rr] : -1;
            }
            float de_r = 0.f, de_w = 0.f;
            for (int c0 = hc * 64; c0 < hc * 64 + 64; c0 += 32) {
                // this block's q, k and G_r - G_m first: one load latency per block
                uint4 q4[4] = {}, k4[4] = {};
                float4 g4[8] = {};
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        q4[i] = __ldg(reinterpret_cast<const uint4 *>(qrow + c0 + 8 * i));
                        k4[i] = __ldg(reinterpret_cast<const uint4 *>(krow + c0 + 8 * i));
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) g4[i] = *reinterpret_cast<const float4 *>(gsr + c0 + 4 * i);
                }
                uint32_t xu[32], xk[32];
                __syncwarp();  // the warp converged for its collective TMEM loads
                tmem_ld32(tmem + lb + c0, xu);
                tmem_ld32(tmem + lb + 128 + c0, xk);
                tmem_wait_ld();
                uint32_t pq[16], pk[16];  // dq and dk of the block, packed bf16 pairs
#pragma unroll
                for (int s16 = 0; s16 < 32; s16 += 16) {
                    float dq[16], dk[16], xg[16];
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        float qv[8], kv[8];
                        unpack8(q4[s16 / 8 + h8], qv);
                        unpack8(k4[s16 / 8 + h8], kv);
                        const float4 ga = g4[s16 / 4 + 2 * h8], gb = g4[s16 / 4 + 2 * h8 + 1];
                        const float gd[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int x = 8 * h8 + jj;
                            // fast exponentials: relative error ~1e-5 at |G_r - G_m| = 64, far below bf16's
                            const float u = __expf(gd[jj]) * __uint_as_float(xu[s16 + x]);
                            const float dK = __expf(-gd[jj]) * __uint_as_float(xk[s16 + x]);
                            dq[x] = e * scale * u;
                            dk[x] = e * dK;
                            xg[x] = qv[jj] * dq[x] - kv[jj] * dk[x];
                            de_r += scale * qv[jj] * u;
                            de_w += kv[jj] * dK;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        pq[s16 / 2 + i] = pack2(dq[2 * i], dq[2 * i + 1]);
                        pk[s16 / 2 + i] = pack2(dk[2 * i], dk[2 * i + 1]);
                    }
                    if (!valid) {
#pragma unroll
                        for (int x = 0; x < 16; ++x) xg[x] = 0.f;
                    }
                    warp_put16(patch, lane, xg, a.dg_c, kKey, c0 + s16, sr);
                    // the block's column sums over this warp's 32 rows, still in
                    // the patch: lane (half, col) adds 16 rows, then the halves meet
                    {
                        const float *pc = patch + (lane >> 4) * 16 * kPatchStride + (lane & 15);
                        float cs = 0.f;
#pragma unroll
                        for (int x = 0; x < 16; ++x) cs += pc[x * kPatchStride];
                        cs += __shfl_xor_sync(0xffffffffu, cs, 16);
                        if (lane < 16) c.csum[quarter * kKey + c0 + s16 + lane] = cs;
                        __syncwarp();  // the patch is rewritten next
                    }
                }
                warp_put32_bf16(patch, lane, pq, dq_c, kKey, c0, sr);
                warp_put32_bf16(patch, lane, pk, dk_c, kKey, c0, sr);
            }
            for (int c0 = hc * (DV / 2); c0 < (hc + 1) * (DV / 2); c0 += 32) {
                uint32_t xv[32];
                __syncwarp();
                tmem_ld32(tmem + lb + 256 + c0, xv);
                tmem_wait_ld();
                uint32_t pv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pv[i] = pack2(__uint_as_float(xv[2 * i]), __uint_as_float(xv[2 * i + 1]));
                warp_put32_bf16(patch, lane, pv, dv_c, DV, c0, sr);
            }
            if (!valid) de_r = de_w = 0.f;
            c.de[(hc * 2) * kRows + erow] = de_r;
            c.de[(hc * 2 + 1) * kRows + erow] = de_w;
        }
        fence_before();
        __syncthreads();
        // router-weight terms of the routed rows: the two column halves, in a fixed order
        if (!r.shared && tid < kRows && tok[tid] >= 0) {
            const int64_t o = (((int64_t)tok[tid] * H + r.h) * topk + sj[tid]) * 2;
            a.de_c[o] = c.de[tid] + c.de[2 * kRows + tid];
            a.de_c[o + 1] = c.de[kRows + tid] + c.de[3 * kRows + tid];
        }
        // the chunk's total of q * dq - k * dk per column: the lane quarters in order
        if (tid >= kRows) {
            const int col = tid - kRows;
            a.dgtot[chunk * kKey + col] =
                ((c.csum[col] + c.csum[kKey + col]) + c.csum[2 * kKey + col]) + c.csum[3 * kKey + col];
        }
        __syncthreads();  // TMEM, the router-weight sums and this metadata buffer are reused
        chunk = next;
        r = rn;
        have = have_next;
        mb ^= 1;
    }
    if (failed) cp_async_wait_all();  // no copy may still be writing shared memory when the CTA exits
    if (failed && tid == 0) atomicOr(a.flags, SSE_DEVICE_TIMEOUT);
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- gate gradient: reverse running sums of q * dq - k * dk over each item ----
// Slot row of every row of a chunk into shared memory (-1 past the item's end).
__device__ __forceinline__ void chunk_slot_rows(const BackwardArgs &a, const ChunkRef &r, int H, int topk, int ncon,
                                                int64_t *srow) {
    if (threadIdx.x < kRows) {
        int t, j;
        float e;
        row_meta(a, r, threadIdx.x, topk, t, e, j);
        srow[threadIdx.x] = t >= 0 ? ((int64_t)t * H + r.h) * ncon + j : -1;
    }
}

// Inside each chunk, from its last row: dg_c = carry + the terms of this and
// every later row, where the chunk's carry is rowsum(S_T * dL/dS_T) plus the
// column totals of the item's later chunks, added from the last chunk down.
__global__ void __launch_bounds__(kKey)
bwd_dg_apply_kernel(BackwardArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared) {
    __shared__ int64_t srow[kRows];
    const int ncon = topk + use_shared;
    for (int64_t chunk = blockIdx.x; chunk < a.num_chunks; chunk += gridDim.x) {
        ChunkRef r;
        if (!locate_chunk(a, chunk, H, N, use_shared, r)) break;
        chunk_slot_rows(a, r, H, topk, ncon, srow);
        const int64_t cb = a.pad_off[r.item] / kRows;
        const int nch = (a.pad_off[r.item + 1] - a.pad_off[r.item]) / kRows;
        float run = a.fterm[(int64_t)r.item * kKey + threadIdx.x];
        for (int j = nch - 1; j > r.n; --j) run += a.dgtot[(cb + j) * kKey + threadIdx.x];
        __syncthreads();
        for (int x0 = kRows - 1; x0 >= 0; x0 -= 8) {  // eight rows' loads ahead of the running sum
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = srow[x0 - i] >= 0 ? a.dg_c[srow[x0 - i] * kKey + threadIdx.x] : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (srow[x0 - i] < 0) continue;
                run += t[i];
                a.dg_c[srow[x0 - i] * kKey + threadIdx.x] = run;
            }
        }
        __syncthreads();
    }
}

template <int DV>
cudaError_t launch_chunked_t(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream, int *launches) {
    const int H = cfg.num_heads, N = cfg.num_partitions, topk = cfg.top_k, us = cfg.use_shared;
    const int nitems = a.num_seqs * H * (N + us);
    static bool attr_set = false;  // benign race: every caller sets the same values
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(bwd_chunk_sums_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)chunk_smem_bytes(5));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_chunk_grads_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)chunk_smem_bytes(6));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaError_t e = cudaMemsetAsync(a.flags, 0, 2 * sizeof(int32_t), stream);
    if (e == cudaSuccess && nitems > 0) e = cudaMemsetAsync(a.marks, 0, sizeof(int32_t) * nitems, stream);
    if (e != cudaSuccess) return e;
    if (nitems > 0) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int grid = (int)std::max<int64_t>(
            1, std::min<int64_t>(a.num_chunks, std::min(sms > 0 ? sms : 148, kBwdScratchCtas)));
        const int grid_dg = (int)std::max<int64_t>(1, std::min<int64_t>(a.num_chunks, 16 * (sms > 0 ? sms : 148)));
        bwd_chunk_sums_kernel<DV><<<grid, kThr, chunk_smem_bytes(5), stream>>>(a, H, N, topk, us, cfg.scale);
        bwd_state_scan_kernel<DV><<<dim3(nitems, kKey * DV / 4 / 256), 256, 0, stream>>>(a, H, N, us);
        bwd_chunk_grads_kernel<DV><<<grid, kThr, chunk_smem_bytes(6), stream>>>(a, H, N, topk, us, cfg.scale);
        bwd_dg_apply_kernel<<<grid_dg, kKey, 0, stream>>>(a, H, N, topk, us);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 4;
        // items whose gates left the factorised form's range: the per-token kernel
        BackwardArgs b = a;
        b.seg_list = a.redo_list;
        b.seg_count = a.flags + 1;
        e = launch_backward_segments(cfg, b, stream);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    e = launch_backward_combine(cfg, a, stream);
    *launches += 1;
    return e;
}

}  // namespace
}  // namespace sse

namespace sse {

bool backward_chunked_supported(const sse_config_t &cfg) {
    return cfg.dtype == SSE_BF16 && cfg.key_dim == kKey && (cfg.value_dim == 64 || cfg.value_dim == 128);
}

cudaError_t launch_backward_chunked(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream,
                                    int *launches) {
    if (!backward_chunked_supported(cfg)) return cudaErrorInvalidValue;
    return cfg.value_dim == 128 ? launch_chunked_t<128>(cfg, a, stream, launches)
                                : launch_chunked_t<64>(cfg, a, stream, launches);
}

}  // namespace sse

#ifdef SSE_FAULT_INJECT
// Checked build only: sets the fault mode read by bwd_chunk_grads_kernel (0 =
// none, 1 = CTA 0 withholds its first product round).  Returns the CUDA error
// of the copy.
extern "C" int sse_debug_set_bwd_fault(int mode) {
    return (int)cudaMemcpyToSymbol(sse::g_bwd_fault_mode, &mode, sizeof(int));
}
#endif
