// delta_chunked.cu -- SSE on the gated delta rule in chunked form on the
// tensor cores, for bf16 tokens and c = d = 128 (the recurrence and its
// reading are those of delta.cu: "Scaling Linear Attention with Sparse State
// Expansion", close-reading notes section 2.1 eq. 6 and section 6; DeltaNet's
// update, "动态线性注意力" section 2.1 eq. 4).
//
// One work item (a routed segment or a shared (sequence, head)) is a sequence
// of rows t with key k_t, value v_t, query factor qf_t = e_t scale, writing
// strength b_t = e_t beta_t and decay alpha_t (e_t: the router weight, 1 for
// the shared partition).  With w_t = k_t S_{t-1} (row vectors, S is c x d):
//   u_t = b_t (v_t - alpha_t w_t),  S_t = alpha_t S_{t-1} + k_t^T u_t,
//   o_t = qf_t q_t S_t.
// In a chunk of 128 rows starting from the state S0, with G_t the running sum
// of log alpha from the chunk's first row through row t, gamma_t = exp(G_t)
// and Gamma_ts = exp(G_t - G_s) (s <= t, so every factor is at most 1):
//   alpha_t w_t = gamma_t k_t S0 + sum_{s<t} Gamma_ts (k_t . k_s) u_s,
// so the chunk's u rows solve a unit lower-triangular system:
//   (I + L) U = diag(b) (V - diag(gamma) K S0),  L_ts = b_t Gamma_ts (k_t . k_s), s < t,
//   U = T R,  T = (I + L)^-1 diag(b),  R = V - diag(gamma) (K S0);
//   O = diag(qf gamma) Q S0 + (tril(Q K^T) . Gamma . qf) U;
//   S_end = gamma_last S0 + (diag(gamma_last / gamma) K)^T U.
// Per chunk, tcgen05 products (K K^T and K S0; Q K^T, waited for later;
// (qf gamma Q) S0; the lower-left quadrant of T; T R; then P U and the state
// update), all issued by one thread, and between them passes over TMEM rows
// and the inverse X of I + L in float32 on the CUDA cores: the diagonal
// 16 x 16 blocks D by forward substitution, each 64-row half by doubling
// (X_10 = -D_1 L_10 D_0 for the four 32-row pairs, then -X_B L_BA X_A for
// each half's 32 x 32 lower-left block).  T = X diag(b) is built as a bf16
// tile whose lower-left 64 x 64 quadrant is -T_BB (M_BA T_AA), M = L without
// its row factor b, two products on the tensor cores.  Gamma_ts is formed as
// exp(G_t - G_m) exp(G_m - G_s) around the chunk's midpoint row m when that
// stays within float32, else per element.  The state stays in TMEM in
// float32 for the whole item; its bf16 copy is the operand of K S0 and Q S0.
// Read-outs go to bf16 partial slots ([T, H, k, d] and [T, H, d], the layout
// of the token-serial kernels' float32 ones) that launch_combine sums in
// float32.
#include <algorithm>

#include "chunk_tiles.cuh"
#include "sse_internal.cuh"
#include "umma.cuh"

namespace sse {
namespace {

using namespace umma;
using namespace tiles;

constexpr int kRows = kChunkRows;  // 128 rows per chunk
constexpr int kC = 128, kD = 128;  // key and value dimensions
constexpr int kThr = 256;          // 8 warps: two per TMEM lane quarter
constexpr uint32_t kTile = 128 * 256;
constexpr int kNB = kRows / 16;               // 16-row blocks of the chunk
constexpr int kRS = 20;                       // floats per stored block row (16 used; rows 16-byte aligned)
constexpr int kBS = 16 * kRS + 4;             // floats per stored 16 x 16 block (+4: consecutive blocks 4 banks apart)
constexpr int kNBlk = kNB * (kNB + 1) / 2;    // lower blocks, diagonal included
// Gamma_ts = exp(G_t - G_s) is formed as exp(G_t - G_m) exp(G_m - G_s) around
// the chunk's midpoint row m when every |G - G_m| of the chunk is at most
// kFacRange (each factor then stays within float32, their product is at most
// 1); a chunk with stronger decay takes one exponential per element.
constexpr int kMidRow = kRows / 2 - 1;
constexpr float kFacRange = 60.f;
#ifdef SSE_FAULT_INJECT
// Checked build (libsse_checked.so, for the failure-detection test only):
// every bounded wait gives up after 50 ms, and g_delta_fault_mode = 1 makes
// CTA 0 issue neither the first product round of its first chunk nor its
// commit, so that the wait on it runs out and the kernel takes its abort path
// (SSE_DEVICE_TIMEOUT, TMEM freed) with no product in flight.
__device__ int g_delta_fault_mode = 0;
constexpr uint64_t kWait = 50000000ull;
#else
constexpr uint64_t kWait = 2000000000ull;
#endif

__device__ __forceinline__ int blkidx(int I, int K) { return I * (I + 1) / 2 + K; }

// Shared memory: five operand tiles from a 1024-aligned base, the lower
// blocks of I + L (then of its inverse), eight scratch blocks for the
// inverse's intermediate products, per-row metadata, the mbarrier and
// the TMEM address slot.  The warps' store patches of the read-out use the
// T / P tile, free by then (the next chunk's rows are landing in Q, K, V).
struct DSmem {
    unsigned char *tQ, *tK, *tV, *tS, *tT;
    float *blk, *zs;
    int *tok, *slotj;
    float *G, *b, *qf, *ec, *red, *patch;
    uint32_t bar, bar2;  // the products' mbarrier; the one of Q K^T (waited for a few phases later)
    uint32_t *tslot;
    int *item;
};
__device__ __forceinline__ DSmem carve(unsigned char *raw) {
    unsigned char *sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    DSmem c;
    c.tQ = sm;
    c.tK = sm + kTile;
    c.tV = sm + 2 * kTile;
    c.tS = sm + 3 * kTile;
    c.tT = sm + 4 * kTile;
    c.blk = reinterpret_cast<float *>(sm + 5 * kTile);  // [kNBlk][kBS]
    c.zs = c.blk + kNBlk * kBS;                          // [kNB][kBS] products inside the doubling stages
    c.tok = reinterpret_cast<int *>(c.zs + kNB * kBS);
    c.slotj = c.tok + kRows;
    c.G = reinterpret_cast<float *>(c.slotj + kRows);
    c.b = c.G + kRows;
    c.qf = c.b + kRows;
    c.ec = c.qf + kRows;    // exp(G_m - G_s) of the chunk's rows s (the column factors of Gamma)
    c.red = c.ec + kRows;   // [8]
    c.patch = reinterpret_cast<float *>(c.tT);  // [8 warps][32][kPatchStride] in the T / P tile
    uint64_t *bar = reinterpret_cast<uint64_t *>(c.red + 8);
    c.bar = smem_u32(bar);
    c.bar2 = smem_u32(bar + 1);
    c.tslot = reinterpret_cast<uint32_t *>(bar + 2);
    c.item = reinterpret_cast<int *>(c.tslot + 1);
    return c;
}
constexpr size_t delta_smem_bytes() {
    return 1024 + 5 * (size_t)kTile + (size_t)(kNBlk + kNB) * kBS * 4 + 2 * kRows * 4 + 4 * kRows * 4 + 8 * 4 + 24 +
           16;
}

// One elected thread (kIssuer: every product and commit of the CTA comes
// from it, and it is outside the row-metadata warps, so that its issue -- which
// waits while the tensor core's queue is full -- delays no other work) issues
// the products and commits them to the CTA's mbarrier; every thread runs
// `during` (work that touches neither the products' operands nor their
// results; false = a failed wait of its own) and then waits (bounded).
// Shared-memory operands written by the generic proxy before the call are
// made visible to the tensor core first.  Returns false, in every thread, when
// a wait ran out.
constexpr int kIssuer = 144;  // warp 4, lane 16
struct NoWork {
    __device__ bool operator()() const { return true; }
};
template <typename F, typename D = NoWork>
__device__ __forceinline__ bool run_mma(const DSmem &c, uint32_t &phase, F issue, bool withhold = false,
                                        D during = D()) {
    fence_proxy_async();
    fence_before();
    __syncthreads();
    if (threadIdx.x == kIssuer && !withhold) {
        fence_after();
        issue();
        commit(c.bar);
    }
    __syncwarp();
    const bool dok = during();
    const bool ok = mbar_wait_bounded(c.bar, phase, kWait) && dok;
    phase ^= 1u;
    fence_after();
    return __syncthreads_and(ok) != 0;
}

// Loads kept where they are written (volatile: the compiler neither sinks them
// towards their use nor merges them), for metadata fetched a phase or a chunk
// before it is needed.
__device__ __forceinline__ int ld_early_s32(const int32_t *p) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_early_f32(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_early_bf16(const __nv_bfloat16 *p) {
    unsigned short u;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(u) : "l"(p));
    return __uint_as_float((uint32_t)u << 16);
}

// L2 prefetch of one 256-byte bf16 row of 128 elements (two 128-byte lines; no
// completion to wait for)
__device__ __forceinline__ void prefetch_row_l2(const __nv_bfloat16 *row) {
    asm volatile("prefetch.global.L2 [%0];" :: "l"(row));
    asm volatile("prefetch.global.L2 [%0];" :: "l"(row + 64));
}

// 8 consecutive bf16 of a tile row (16 bytes) <-> float32
__device__ __forceinline__ void ld8(const unsigned char *p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void st8(unsigned char *p, const float (&f)[8]) {
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__global__ void __launch_bounds__(kThr, 1)
delta_chunked_kernel(DeltaArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared, float scale,
                     int32_t num_items, int32_t *flags) {
    extern __shared__ unsigned char smem_raw[];
    const DSmem c = carve(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // TMEM lane quarter (warp % 4) = rows, column half = warp / 4
    const int quarter = warp & 3, hc = warp >> 2, erow = 32 * quarter + lane;
    const uint32_t lb = (uint32_t)(32 * quarter) << 16;
    if (warp == 0) tmem_alloc(smem_u32(c.tslot), 512);
    if (tid == 0) {
        mbar_init(c.bar, 1);
        mbar_init(c.bar2, 1);
        mbar_fence_init();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *c.tslot;
    const uint32_t tA1 = tmem, tA2 = tmem + 128, tO = tmem + 256, tSt = tmem + 384;
    uint32_t phase = 0, phase2 = 0;
    bool failed = false, a2pend = false;  // a2pend: a chunk's Q K^T committed and not yet waited for
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q), *k = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *qs = static_cast<const __nv_bfloat16 *>(a.qs), *ks = static_cast<const __nv_bfloat16 *>(a.ks);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
    const __nv_bfloat16 *la = static_cast<const __nv_bfloat16 *>(a.log_alpha);
    const __nv_bfloat16 *bt = static_cast<const __nv_bfloat16 *>(a.beta);
    const int nshared = use_shared ? a.num_seqs * H : 0;
    const int P = N + use_shared;
    int32_t *counter = flags + 1;
    float *patch = c.patch + warp * 32 * kPatchStride;
#ifdef SSE_FAULT_INJECT
    bool first_chunk = true;  // of this CTA (the checked build's fault switch)
#endif

    for (;;) {
        if (tid == 0) *c.item = atomicAdd(counter, 1);
        __syncthreads();
        const int item = *c.item;
        __syncthreads();  // the slot is written again by the next claim
        if (item >= num_items) break;
        int b, h, slot, base, len;
        const bool shared = item < nshared;
        if (shared) {
            b = item / H;
            h = item % H;
            slot = N;
            base = a.cu_seqlens[b];
            len = a.cu_seqlens[b + 1] - base;
        } else {
            const int s = item - nshared;
            slot = s % N;
            h = (s / N) % H;
            b = s / (N * H);
            base = a.seg_off[s];
            len = a.seg_off[s + 1] - base;
        }
        const int64_t state_off = (((int64_t)b * H + h) * P + slot) * (int64_t)kC * kD;
        if (len == 0) {
            // nothing to apply: the final state is the initial one
            if (a.final_state && a.final_state != a.init)
                for (int x = tid; x < kC * kD / 4; x += kThr)
                    reinterpret_cast<float4 *>(a.final_state + state_off)[x] =
                        a.init ? reinterpret_cast<const float4 *>(a.init + state_off)[x]
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        const __nv_bfloat16 *qsrc = shared && qs ? qs : q, *ksrc = shared && ks ? ks : k;
        // the initial state into TMEM (row = lane of the quarter, this warp's column half)
        for (int g = 0; g < 2; ++g) {
            const int col0 = 64 * hc + 32 * g;
            uint32_t x[32];
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                if (a.init)
                    y = *reinterpret_cast<const float4 *>(a.init + state_off + (int64_t)erow * kD + col0 + 4 * i4);
                x[4 * i4] = __float_as_uint(y.x);
                x[4 * i4 + 1] = __float_as_uint(y.y);
                x[4 * i4 + 2] = __float_as_uint(y.z);
                x[4 * i4 + 3] = __float_as_uint(y.w);
            }
            __syncwarp();
            tmem_st32(tSt + lb + col0, x);
        }
        tmem_wait_st();

        // Row tid's metadata, fetched ahead in two steps so that no warp waits
        // on a dependent load: the grouped record two chunks ahead, then (a
        // chunk later, while the first products run) the token's router weight,
        // gates and an L2 prefetch of its q, k, v rows, which the copies of
        // prepare then find in L2.
        int nrec = 0, nt = -1, njj = 0;
        float ne = 0.f, nbeta = 0.f, nlg = 0.f;
        auto fetch_rec = [&](int ch) {
            const int idx = ch * kRows + tid;
            if (!shared && tid < kRows && idx < len) nrec = ld_early_s32(a.perm_rec + base + idx);
        };
        auto fetch_rest = [&](int ch) {
            const int idx = ch * kRows + tid;
            nt = -1;
            njj = 0;
            ne = nbeta = nlg = 0.f;
            if (tid < kRows && idx < len) {
                if (shared) {
                    nt = base + idx;
                    ne = 1.f;
                } else {
                    nt = nrec / topk;
                    njj = nrec - nt * topk;
                    ne = ld_early_f32(a.topk_w + ((int64_t)nt * H + h) * topk + njj);
                }
                const int64_t th = (int64_t)nt * H + h;
                nlg = ld_early_bf16(la + th);
                nbeta = ld_early_bf16(bt + th);
                prefetch_row_l2(qsrc + th * kC);
                prefetch_row_l2(ksrc + th * kC);
                prefetch_row_l2(v + th * kD);
            }
        };
        // row metadata (fetched ahead) and the running log-decay G (inclusive)
        // of chunk ch, then its q, k, v rows by asynchronous copies (waited for
        // before products 1)
        auto prepare = [&](int ch) {
            __syncthreads();  // every reader of the metadata and of the Q, K, V tiles is done
            float lg = 0.f;
            if (tid < kRows) {
                c.tok[tid] = nt;
                c.slotj[tid] = njj;
                c.b[tid] = ne * nbeta;
                c.qf[tid] = ne * scale;
                lg = nlg;
            }
            // inclusive scan of lg over rows 0..127 (warps 0..3)
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, lg, o);
                if (lane >= o) lg += y;
            }
            if (lane == 31) c.red[warp] = lg;  // warps 4..7 write zeros: red[7] starts clear
            __syncthreads();
            if (tid < kRows) {
                for (int w2 = 0; w2 < warp; ++w2) lg += c.red[w2];
                c.G[tid] = lg;
            }
            __syncthreads();
            if (tid < kRows) {  // read after the next barrier, with red[7]'s range flag (zeroed by the scan)
                const float dG = c.G[kMidRow] - c.G[tid];
                c.ec[tid] = __expf(dG);
                if (!(fabsf(dG) <= kFacRange)) c.red[7] = 1.f;
            }
            stage_rows_n<128, 3>({c.tQ, c.tK, c.tV}, {qsrc, ksrc, v}, c.tok, H, h);
        };
        const int nch = (len + kRows - 1) / kRows;
        fetch_rec(0);
        fetch_rest(0);
        prepare(0);
        if (nch > 1) fetch_rec(1);
        for (int ch = 0; ch < nch; ++ch) {
            // ---- the state's bf16 copy and the decay of the chunk, while the rows land ----
            {
                const float gC = __expf(c.G[kRows - 1]);
                for (int g = 0; g < 2; ++g) {
                    const int col0 = 64 * hc + 32 * g;
                    uint32_t x[32];
                    __syncwarp();
                    tmem_ld32(tSt + lb + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(x[8 * j8 + i]);
                        st8(c.tS + toff(erow, col0 + 8 * j8), f);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __float_as_uint(gC * __uint_as_float(x[i]));
                    tmem_st32(tSt + lb + col0, x);
                }
                tmem_wait_st();
            }
            cp_async_wait_all();
            // ---- products 1: A1 = K K^T, Y = K S0, waited for now; A2 = Q K^T on the second
            //      mbarrier, waited for before the P pass (the raw Q tile stays untouched) ----
#ifdef SSE_FAULT_INJECT
            const bool withhold = g_delta_fault_mode == 1 && blockIdx.x == 0 && first_chunk;
            first_chunk = false;
#else
            const bool withhold = false;
#endif
            bool ok = run_mma(c, phase, [&] {
                constexpr uint32_t idT = idesc_bf16(128, 128, 0, 0), idS = idesc_bf16(128, kD, 0, 1);
                for (int k16 = 0; k16 < kC; k16 += 16) {
                    const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2, ro = (k16 / 8) * 2048;
                    mma_bf16(tA1, desc_sw128(smem_u32(c.tK) + ko, 16, 2048), desc_sw128(smem_u32(c.tK) + ko, 16, 2048),
                             idT, k16 > 0);
                    mma_bf16(tO, desc_sw128(smem_u32(c.tK) + ko, 16, 2048), desc_sw128(smem_u32(c.tS) + ro, 1024, 2048),
                             idS, k16 > 0);
                }
            }, withhold, [&] {
                if (ch + 1 < nch) fetch_rest(ch + 1);  // uses the record fetched a chunk ago
                if (ch + 2 < nch) fetch_rec(ch + 2);
                return true;
            });
            if (ok && tid == kIssuer && !withhold) {  // A2, queued behind nothing: it runs under the pass below
                fence_after();
                constexpr uint32_t idT = idesc_bf16(128, 128, 0, 0);
                for (int k16 = 0; k16 < kC; k16 += 16) {
                    const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                    mma_bf16(tA2, desc_sw128(smem_u32(c.tQ) + ko, 16, 2048), desc_sw128(smem_u32(c.tK) + ko, 16, 2048),
                             idT, k16 > 0);
                }
                commit(c.bar2);
            }
            a2pend = ok && !withhold;
            if (!ok) {
                failed = true;
                break;
            }
            // ---- L blocks from A1; R = V - gamma Y in place of V; Q scaled by qf gamma into the T tile ----
            const float Gm = c.G[kMidRow];
            const bool fac = c.red[7] == 0.f;  // every |G - G_m| of the chunk within kFacRange (uniform)
            {
                const int t = erow;
                const float Gt = c.G[t], bt_ = c.b[t], gt = __expf(Gt), qg = c.qf[t] * gt;
                const float erm = __expf(Gt - Gm), ber = bt_ * erm;  // exp(G_t - G_m), b_t exp(G_t - G_m)
                for (int g = 0; g < 2; ++g) {
                    const int col0 = 64 * hc + 32 * g;
                    uint32_t x[32];
                    __syncwarp();
                    tmem_ld32(tA1 + lb + col0, x);
                    tmem_wait_ld();
                    // row t of the lower blocks, four columns per 16-byte store (rows of
                    // a warp 80 bytes apart: conflict-free); the entries on and above the
                    // diagonal of a diagonal block are written as zeros (never read).  The
                    // lower-left quadrant (t >= 64, s < 64) holds M_ts = Gamma_ts (k_t . k_s),
                    // L without its row factor b_t: only the quadrant's products read it.
                    float *lrow = c.blk + (t & 15) * kRS;
                    const bool mq = t >= 64 && col0 < 64;  // uniform in the warp
                    const float rf = mq ? erm : ber, bf_ = mq ? 1.f : bt_;
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const int s0 = col0 + 4 * i4;
                        if ((s0 >> 4) > (t >> 4)) continue;  // a block above the diagonal: not stored
                        float l[4];
                        if (fac) {
                            const float4 e4 = *reinterpret_cast<const float4 *>(c.ec + s0);
                            const float es[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) l[i] = s0 + i < t ? rf * es[i] * __uint_as_float(x[4 * i4 + i]) : 0.f;
                        } else {
                            const float4 g4 = *reinterpret_cast<const float4 *>(c.G + s0);
                            const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                l[i] = s0 + i < t ? bf_ * __expf(Gt - gs[i]) * __uint_as_float(x[4 * i4 + i]) : 0.f;
                        }
                        *reinterpret_cast<float4 *>(lrow + blkidx(t >> 4, s0 >> 4) * kBS + (s0 & 15)) =
                            make_float4(l[0], l[1], l[2], l[3]);
                    }
                    __syncwarp();
                    tmem_ld32(tO + lb + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        float f[8];
                        unsigned char *pv = c.tV + toff(t, col0 + 8 * j8);
                        ld8(pv, f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] -= gt * __uint_as_float(x[8 * j8 + i]);
                        st8(pv, f);
                        ld8(c.tQ + toff(t, col0 + 8 * j8), f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] *= qg;
                        st8(c.tT + toff(t, col0 + 8 * j8), f);
                    }
                }
            }
            // ---- products 2a, issued now and waited for after the inverse: Z = (qf gamma Q) S0 into O ----
            fence_proxy_async();
            fence_before();
            __syncthreads();
            if (tid == kIssuer) {
                fence_after();
                constexpr uint32_t idS = idesc_bf16(128, kD, 0, 1);
                for (int k16 = 0; k16 < kC; k16 += 16) {
                    const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2, ro = (k16 / 8) * 2048;
                    mma_bf16(tO, desc_sw128(smem_u32(c.tT) + ko, 16, 2048), desc_sw128(smem_u32(c.tS) + ro, 1024, 2048),
                             idS, k16 > 0);
                }
                commit(c.bar);
            }
            // ---- the inverse of I + L: diagonal blocks, one warp each (lanes 0..15, one
            //      column each; lane 16 of warp 4 is the issuer, still queueing products 2a) ----
            if (lane < 16) {
                float *bd = c.blk + blkidx(warp, warp) * kBS;
                float x[16];  // column `lane` of the block's inverse
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = r == lane ? 1.f : 0.f;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int kk = 0; kk < r; ++kk) acc = fmaf(bd[r * kRS + kk], x[kk], acc);
                    if (r > lane) x[r] = -acc;  // rows above the diagonal keep 0, the diagonal 1
                }
                __syncwarp(0x0000ffffu);  // every read of the block's L is done
#pragma unroll
                for (int r = 0; r < 16; ++r) bd[r * kRS + lane] = x[r];
            }
            __syncthreads();
            // ---- each 64-row half from its diagonal blocks D, by doubling ----
            // (A) the four 32-row pairs: X[2p+1][2p] = -D[2p+1] (L[2p+1][2p] D[2p]);
            // (B) in each half (blocks B0..B0+3) the 32 x 32 lower-left block:
            //     X_BA = -X_B (L_BA X_A), X_A, X_B the pairs' 32-row inverses.
            // Every stage keeps all 256 threads busy on a register tile of four
            // columns (one or two rows), reading 16-byte vectors: the left
            // factor's row and the right factor's rows; the intermediate products
            // go to the scratch blocks.  The lower block storage of a pair (the
            // one of X_A, X_B) is zero above its block diagonal, so those terms
            // are skipped.
            {
                auto ld4 = [&](const float *p) { return *reinterpret_cast<const float4 *>(p); };
                auto fma4 = [&](float a, const float4 &x, float (&acc)[4]) {
                    acc[0] = fmaf(a, x.x, acc[0]);
                    acc[1] = fmaf(a, x.y, acc[1]);
                    acc[2] = fmaf(a, x.z, acc[2]);
                    acc[3] = fmaf(a, x.w, acc[3]);
                };
                // acc += row (16 values at lrow) times the 16 x 4 column strip at rcol (rows kRS apart)
                // (all loads issued before the products: one round of shared-memory latency)
                auto strip = [&](const float *lrow, const float *rcol, float (&acc)[4]) {
                    float4 l[4], x[16];
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) l[m4] = ld4(lrow + 4 * m4);
#pragma unroll
                    for (int m = 0; m < 16; ++m) x[m] = ld4(rcol + m * kRS);
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        fma4(l[m4].x, x[4 * m4], acc);
                        fma4(l[m4].y, x[4 * m4 + 1], acc);
                        fma4(l[m4].z, x[4 * m4 + 2], acc);
                        fma4(l[m4].w, x[4 * m4 + 3], acc);
                    }
                };
                // the same for two rows sharing the strip (each strip vector read once)
                auto strip2 = [&](const float *lrow0, const float *lrow1, const float *rcol, float (&acc0)[4],
                                  float (&acc1)[4]) {
                    float4 l0[4], l1[4], x[16];
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        l0[m4] = ld4(lrow0 + 4 * m4);
                        l1[m4] = ld4(lrow1 + 4 * m4);
                    }
#pragma unroll
                    for (int m = 0; m < 16; ++m) x[m] = ld4(rcol + m * kRS);
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        const float a0[4] = {l0[m4].x, l0[m4].y, l0[m4].z, l0[m4].w};
                        const float a1[4] = {l1[m4].x, l1[m4].y, l1[m4].z, l1[m4].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            fma4(a0[i], x[4 * m4 + i], acc0);
                            fma4(a1[i], x[4 * m4 + i], acc1);
                        }
                    }
                };
                auto st4 = [&](float *p, const float (&v)[4], float sgn) {
                    *reinterpret_cast<float4 *>(p) = make_float4(sgn * v[0], sgn * v[1], sgn * v[2], sgn * v[3]);
                };
                {
                    // (A) thread: pair P, row rr, columns 4 c4 .. 4 c4 + 3
                    const int P = tid >> 6, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
                    float *lo = c.blk + blkidx(2 * P + 1, 2 * P) * kBS;
                    float *w = c.zs + P * kBS;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    strip(lo + rr * kRS, c.blk + blkidx(2 * P, 2 * P) * kBS + c4, acc);  // L D[2p]
                    st4(w + rr * kRS + c4, acc, 1.f);
                    __syncthreads();
                    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
                    strip(c.blk + blkidx(2 * P + 1, 2 * P + 1) * kBS + rr * kRS, w + c4, acc2);  // D[2p+1] W
                    st4(lo + rr * kRS + c4, acc2, -1.f);
                    __syncthreads();
                }
                {
                    // (B) thread: half h, rows r of blocks B0+2 and B0+3, columns cj .. cj+3
                    // of block column B0 + jb (a warp shares jb)
                    const int h2 = tid >> 7, u = tid & 127, r = u & 15, c4 = u >> 4, jb = c4 >> 2, cj = (c4 & 3) * 4;
                    const int B0 = 4 * h2;
                    float *w = c.zs + 4 * h2 * kBS;  // W[i][j], i, j in {0, 1}: block 2 i + j
                    {
                        float a2[4] = {0.f, 0.f, 0.f, 0.f}, a3[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb) {
                            if (kb < jb) continue;  // X_A's block (0, 1) is zero
                            strip2(c.blk + blkidx(B0 + 2, B0 + kb) * kBS + r * kRS,
                                   c.blk + blkidx(B0 + 3, B0 + kb) * kBS + r * kRS,
                                   c.blk + blkidx(B0 + kb, B0 + jb) * kBS + cj, a2, a3);
                        }
                        st4(w + jb * kBS + r * kRS + cj, a2, 1.f);
                        st4(w + (2 + jb) * kBS + r * kRS + cj, a3, 1.f);
                    }
                    __syncthreads();
                    {
                        // X_B's block (0, 1) is zero: row block 2 takes W[0] only
                        float a2[4] = {0.f, 0.f, 0.f, 0.f}, a3[4] = {0.f, 0.f, 0.f, 0.f};
                        const float *w0 = w + jb * kBS + cj, *w1 = w + (2 + jb) * kBS + cj;
                        strip2(c.blk + blkidx(B0 + 2, B0 + 2) * kBS + r * kRS,
                               c.blk + blkidx(B0 + 3, B0 + 2) * kBS + r * kRS, w0, a2, a3);
                        strip(c.blk + blkidx(B0 + 3, B0 + 3) * kBS + r * kRS, w1, a3);
                        st4(c.blk + blkidx(B0 + 2, B0 + jb) * kBS + r * kRS + cj, a2, -1.f);
                        st4(c.blk + blkidx(B0 + 3, B0 + jb) * kBS + r * kRS + cj, a3, -1.f);
                    }
                    // read by the quadrant after its first barrier
                }
            }
            // ---- T = X diag(b) as the bf16 tile of U = T R (rows t, columns s), its lower-left
            //      quadrant on the tensor cores ----
            // With L_BA = diag(b_B) M_BA, the quadrant of T is
            //   T_BA = X_BA diag(b_A) = -X_B L_BA X_A diag(b_A) = -T_BB (M_BA T_AA):
            // T_AA = X_A diag(b_A) and T_BB = X_B diag(b_B) go to their places in the
            // T tile (the upper-right quadrant zero), M_BA to the state tile (free:
            // products 2a are done); W = M_BA T_AA (T_AA read in place as the
            // MN-major B operand) into TMEM columns 0..63, W back to the state tile,
            // then T_BB W with the T tile's columns 64..127 as the A operand (its
            // rows 0..63 are the zero quadrant), rows 64..127 of TMEM columns
            // 64..127, negated into the lower-left quadrant.  Rows 64..127 of the
            // first product's A operand only feed output rows that are never read.
            {
                const bool zok = mbar_wait_bounded(c.bar, phase, kWait);
                phase ^= 1u;
                fence_after();
                if (!__syncthreads_and(zok)) {
                    failed = true;
                    break;
                }
                // element (row, col) of the lower block storage (zero above the block diagonal)
                auto ld8f = [&](int row, int col, float (&f)[8]) {
                    if ((row >> 4) < (col >> 4)) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = 0.f;
                        return;
                    }
                    const float *p = c.blk + blkidx(row >> 4, col >> 4) * kBS + (row & 15) * kRS + (col & 15);
                    const float4 x0 = *reinterpret_cast<const float4 *>(p), x1 = *reinterpret_cast<const float4 *>(p + 4);
                    f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w;
                    f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
                };
                auto scale_b = [&](int col, float (&f)[8]) {
                    const float4 b0 = *reinterpret_cast<const float4 *>(c.b + col);
                    const float4 b1 = *reinterpret_cast<const float4 *>(c.b + col + 4);
                    f[0] *= b0.x; f[1] *= b0.y; f[2] *= b0.z; f[3] *= b0.w;
                    f[4] *= b1.x; f[5] *= b1.y; f[6] *= b1.z; f[7] *= b1.w;
                };
                const int er = tid >> 2, ec = (tid & 3) * 16;  // this thread's row and 16 columns of a 64 x 64 quadrant
#pragma unroll
                for (int h8 = 0; h8 < 16; h8 += 8) {
                    const int cq = ec + h8;
                    float f[8];
                    ld8f(64 + er, cq, f);  // M_BA: A operand, K-major
                    st8(c.tS + toff(er, cq), f);
                    ld8f(er, cq, f);  // T_AA
                    scale_b(cq, f);
                    st8(c.tT + toff(er, cq), f);
                    ld8f(64 + er, 64 + cq, f);  // T_BB
                    scale_b(64 + cq, f);
                    st8(c.tT + toff(64 + er, 64 + cq), f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) f[i] = 0.f;
                    st8(c.tT + toff(er, 64 + cq), f);  // T_AB = 0
                }
                ok = run_mma(c, phase, [&] {
                    constexpr uint32_t id = idesc_bf16(128, 64, 0, 1);
                    for (int k16 = 0; k16 < 64; k16 += 16)
                        mma_bf16(tA1, desc_sw128(smem_u32(c.tS) + k16 * 2, 16, 2048),
                                 desc_sw128(smem_u32(c.tT) + (k16 / 8) * 2048, 1024, 2048), id, k16 > 0);
                });
                if (!ok) {
                    failed = true;
                    break;
                }
                // W (rows 0..63 of TMEM columns 0..63) into the state tile as the B operand
                if (quarter < 2) {
                    uint32_t x[32];
                    const int col0 = 32 * hc;
                    tmem_ld32(tA1 + lb + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(x[8 * j8 + i]);
                        st8(c.tS + toff(erow, col0 + 8 * j8), f);
                    }
                }
                ok = run_mma(c, phase, [&] {
                    constexpr uint32_t id = idesc_bf16(128, 64, 0, 1);
                    for (int k16 = 0; k16 < 64; k16 += 16)
                        mma_bf16(tA1 + 64, desc_sw128(smem_u32(c.tT) + 1024 + k16 * 2, 16, 2048),
                                 desc_sw128(smem_u32(c.tS) + (k16 / 8) * 2048, 1024, 2048), id, k16 > 0);
                });
                if (!ok) {
                    failed = true;
                    break;
                }
                // T_BA = -(T_BB W) into the lower-left quadrant of the T tile
                if (quarter >= 2) {
                    uint32_t x[32];
                    const int col0 = 32 * hc;
                    tmem_ld32(tA1 + lb + 64 + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = -__uint_as_float(x[8 * j8 + i]);
                        st8(c.tT + toff(erow, col0 + 8 * j8), f);
                    }
                }
            }
            // ---- products 2b: U = T R ----
            ok = run_mma(c, phase, [&] {
                constexpr uint32_t idS = idesc_bf16(128, kD, 0, 1);
                for (int k16 = 0; k16 < kRows; k16 += 16) {
                    const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2, ro = (k16 / 8) * 2048;
                    mma_bf16(tA1, desc_sw128(smem_u32(c.tT) + ko, 16, 2048), desc_sw128(smem_u32(c.tV) + ro, 1024, 2048),
                             idS, k16 > 0);
                }
            }, false, [&] {  // A2 = Q K^T (long done by now) for the P pass below
                const bool a2ok = mbar_wait_bounded(c.bar2, phase2, kWait);
                if (a2ok) {
                    phase2 ^= 1u;
                    a2pend = false;
                }
                return a2ok;
            });
            if (!ok) {
                failed = true;
                break;
            }
            // ---- U -> bf16 in place of R; P = tril(Q K^T) Gamma qf in place of T; K scaled by
            //      gamma_last / gamma in place ----
            {
                const int t = erow;
                const float Gt = c.G[t], qft = c.qf[t], GC = c.G[kRows - 1];
                const float kf = __expf(GC - Gt);
                const float qer = qft * __expf(Gt - Gm);  // qf_t exp(G_t - G_m)
                for (int g = 0; g < 2; ++g) {
                    const int col0 = 64 * hc + 32 * g;
                    uint32_t x[32];
                    __syncwarp();
                    tmem_ld32(tA1 + lb + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(x[8 * j8 + i]);
                        st8(c.tV + toff(t, col0 + 8 * j8), f);
                    }
                    __syncwarp();
                    tmem_ld32(tA2 + lb + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        float f[8];
                        if (fac) {
                            const float4 e0 = *reinterpret_cast<const float4 *>(c.ec + col0 + 8 * j8);
                            const float4 e1 = *reinterpret_cast<const float4 *>(c.ec + col0 + 8 * j8 + 4);
                            const float es[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int s = col0 + 8 * j8 + i;
                                f[i] = s <= t ? qer * es[i] * __uint_as_float(x[8 * j8 + i]) : 0.f;
                            }
                        } else {
                            const float4 g0 = *reinterpret_cast<const float4 *>(c.G + col0 + 8 * j8);
                            const float4 g1 = *reinterpret_cast<const float4 *>(c.G + col0 + 8 * j8 + 4);
                            const float gs[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int s = col0 + 8 * j8 + i;
                                f[i] = s <= t ? qft * __expf(Gt - gs[i]) * __uint_as_float(x[8 * j8 + i]) : 0.f;
                            }
                        }
                        st8(c.tT + toff(t, col0 + 8 * j8), f);
                        unsigned char *pk = c.tK + toff(t, col0 + 8 * j8);
                        ld8(pk, f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] *= kf;
                        st8(pk, f);
                    }
                }
            }
            // ---- products 3: O += P U, S += (K gamma_last / gamma)^T U ----
            ok = run_mma(c, phase, [&] {
                constexpr uint32_t idP = idesc_bf16(128, kD, 0, 1), idU = idesc_bf16(128, kD, 1, 1);
                for (int k16 = 0; k16 < kRows; k16 += 16) {
                    const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2, ro = (k16 / 8) * 2048;
                    mma_bf16(tO, desc_sw128(smem_u32(c.tT) + ko, 16, 2048), desc_sw128(smem_u32(c.tV) + ro, 1024, 2048),
                             idP, 1);
                    mma_bf16(tSt, desc_sw128(smem_u32(c.tK) + ro, 1024, 2048),
                             desc_sw128(smem_u32(c.tV) + ro, 1024, 2048), idU, 1);
                }
            });
            if (!ok) {
                failed = true;
                break;
            }
            // ---- read-out: rows of O to the partial slots, while the next chunk's rows land ----
            {
                int64_t sr[4];  // slot rows this lane stores (-1 past the item's end)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int rr = 32 * quarter + (lane >> 2) + 8 * kk, tt = c.tok[rr];
                    const int64_t th = (int64_t)tt * H + h;
                    sr[kk] = tt < 0 ? -1 : shared ? th : th * topk + c.slotj[rr];
                }
                if (ch + 1 < nch) prepare(ch + 1);
                // bf16 partial rows (the combine sums them in float32)
                __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(shared ? a.part_shared : a.part_routed);
                for (int g = 0; g < 2; ++g) {
                    const int col0 = 64 * hc + 32 * g;
                    uint32_t x[32], w[16];
                    __syncwarp();
                    tmem_ld32(tO + lb + col0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
                    warp_put32_bf16(patch, lane, w, dst, kD, col0, sr);
                }
            }
            fence_before();
        }
        if (failed) break;
        // ---- the final state out of TMEM ----
        __syncthreads();
        fence_after();
        if (a.final_state) {
            for (int g = 0; g < 2; ++g) {
                const int col0 = 64 * hc + 32 * g;
                uint32_t x[32];
                __syncwarp();
                tmem_ld32(tSt + lb + col0, x);
                tmem_wait_ld();
                float *row = a.final_state + state_off + (int64_t)erow * kD + col0;
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4)
                    reinterpret_cast<float4 *>(row)[i4] =
                        make_float4(__uint_as_float(x[4 * i4]), __uint_as_float(x[4 * i4 + 1]),
                                    __uint_as_float(x[4 * i4 + 2]), __uint_as_float(x[4 * i4 + 3]));
            }
        }
        fence_before();
        __syncthreads();  // TMEM's state columns are loaded again by the next item
        fence_after();
    }
    if (failed) cp_async_wait_all();  // no copy may still be writing shared memory when the CTA exits
    if (failed && a2pend) (void)mbar_wait_bounded(c.bar2, phase2, kWait);  // nor a product TMEM when it is freed
    if (failed && tid == 0) atomicOr(flags, SSE_DEVICE_TIMEOUT);
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool delta_chunked_supported(const sse_config_t &cfg) {
    return cfg.dtype == SSE_BF16 && cfg.key_dim == kC && cfg.value_dim == kD;
}

cudaError_t launch_delta_chunked(const sse_config_t &cfg, const DeltaArgs &a, cudaStream_t stream) {
    int32_t *flags = a.flags;
    if (!flags) return cudaErrorInvalidValue;
    static bool attr_set = false;  // benign race: every caller sets the same value
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(delta_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)delta_smem_bytes());
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int nitems = a.num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    cudaError_t e = cudaMemsetAsync(flags, 0, 2 * sizeof(int32_t), stream);
    if (e != cudaSuccess || nitems == 0) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = std::max(1, std::min(nitems, sms > 0 ? sms : 148));
    delta_chunked_kernel<<<grid, kThr, delta_smem_bytes(), stream>>>(a, cfg.num_heads, cfg.num_partitions,
                                                                     cfg.top_k, cfg.use_shared, cfg.scale, nitems,
                                                                     flags);
    return cudaGetLastError();
}

}  // namespace sse

#ifdef SSE_FAULT_INJECT
// Checked build only: sets the fault mode read by delta_chunked_kernel (0 =
// none, 1 = CTA 0 withholds its first product round).  Returns the CUDA error
// of the copy.
extern "C" int sse_debug_set_delta_fault(int mode) {
    return (int)cudaMemcpyToSymbol(sse::g_delta_fault_mode, &mode, sizeof(int));
}
#endif
