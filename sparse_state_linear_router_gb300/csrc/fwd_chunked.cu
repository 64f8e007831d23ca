// fwd_chunked.cu -- tensor-core (tcgen05 + TMEM) chunked SSE forward.
//
// "Scaling Linear Attention with Sparse State Expansion", eqs. 13-14 on the
// grouped per-partition subsequences of the varlen schedule (section 2.6)
// plus the always-on shared partition (section 2.5).  Inside one segment the
// recurrence is gated linear attention with keys e_s k_s, read weights
// e_t * scale and the diagonal gate exp(g); it is evaluated in chunks of
// C = 128 rows.  With G_r the running sum of g inside the chunk (rows
// 0..r) and m the midpoint row (63):
//
//   Qt_r = e_r scale q_r * exp(G_r - G_m)       Kt_s = e_s k_s * exp(G_m - G_s)
//   A    = Qt Kt^T, causally masked (s <= r) -> P (bf16)
//   O    = Qt (exp(G_m) * S) + P V                   (inter- + intra-chunk)
//   S'   = exp(G_last) * S + exp(G_last - G_m) * Kt^T V   (state pass)
//
// Every factor exp(+-(G_r - G_m)) is bounded by exp(|G| over half a chunk),
// which is why the chunk is split at its midpoint.  The state S (c x d,
// fp32) lives in TMEM for the whole segment as S = p * S_stored with a
// per-row pending scale p: each chunk rescales S_stored by exp(G_m) * p in
// place (also producing the bf16 copy used by Qt S), lets the tensor core
// accumulate Kt^T V into it, and sets p = exp(G_last - G_m).
//
// One CTA per segment (routed (b,h,i) or shared (b,h); shared first as they
// are the longest); 8 warps.  Per chunk: all threads build Qt, Kt, V in
// shared memory (128B-swizzled, see umma.cuh); the state rows are rescaled
// from TMEM; thread 0 issues A = Qt Kt^T, S += Kt^T V and O = Qt S'; the
// threads turn A into the masked bf16 P; thread 0 issues O += P V; the
// threads write O (already e-weighted) as the segment's fp32 partial rows.
// Waits on the tensor core are bounded; a timeout sets SSE_DEVICE_TIMEOUT
// in the flags word and the CTA stops after releasing its TMEM.
#include "sse_internal.cuh"
#include "umma.cuh"

namespace sse {
namespace {

using namespace umma;

constexpr int kC = 128;          // chunk rows
constexpr int kThreads = 256;    // 8 warps, two warpgroups
constexpr int kMid = kC / 2 - 1; // midpoint row of the decay split
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
// |G_r - G_m| limit in log2 units (~ 80 in natural-log units)
constexpr float kGateRangeLog2 = 80.f * kLog2e;

constexpr uint32_t kTile = 128 * 256;   // one 128 x 128 bf16 tile: 32 KB

// Shared-memory layout (offsets from a 1024-aligned base).
struct Smem {
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t K = Q + kTile;
    static constexpr uint32_t V = K + kTile;
    static constexpr uint32_t P = V + kTile;
    static constexpr uint32_t S = P + kTile;
    static constexpr uint32_t TOT = S + kTile;            // [33][128] f32 block prefixes; row 32: G_m
    static constexpr uint32_t FMID = TOT + 33 * 128 * 4;  // [128] exp(G_m) per key row
    static constexpr uint32_t BETA = FMID + 128 * 4;      // [128] exp(G_last - G_m)
    static constexpr uint32_t TOK = BETA + 128 * 4;       // [128] int token index (-1: padding)
    static constexpr uint32_t EW = TOK + 128 * 4;         // [128] float e weight
    static constexpr uint32_t DST = EW + 128 * 4;         // [128] int64 partial row offset
    static constexpr uint32_t BAR = DST + 128 * 8;        // 2 mbarriers
    static constexpr uint32_t SLOT = BAR + 16;            // TMEM base address
    static constexpr uint32_t MISC = SLOT + 16;           // abort flag
    static constexpr uint32_t END = MISC + 16;
};
constexpr size_t kSmemBytes = Smem::END + 1024;  // + alignment slack

constexpr uint32_t kTmemA = 0, kTmemO = 128, kTmemS = 256, kTmemCols = 512;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Stores 8 consecutive bf16 columns (one 16-byte chunk) of row `row` of a
// swizzled tile.
__device__ __forceinline__ void st_tile8(unsigned char *tile, int row, int col, uint4 v) {
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, col, 2)) = v;
}

template <int KC, int DV>
__global__ void __launch_bounds__(kThreads, 1)
chunked_segment_kernel(ForwardArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared,
                       float scale) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *sQ = sm + Smem::Q, *sK = sm + Smem::K, *sV = sm + Smem::V;
    unsigned char *sP = sm + Smem::P, *sS = sm + Smem::S;
    float *s_tot = reinterpret_cast<float *>(sm + Smem::TOT);
    float *s_fmid = reinterpret_cast<float *>(sm + Smem::FMID);
    float *s_beta = reinterpret_cast<float *>(sm + Smem::BETA);
    int *s_tok = reinterpret_cast<int *>(sm + Smem::TOK);
    float *s_e = reinterpret_cast<float *>(sm + Smem::EW);
    long long *s_dst = reinterpret_cast<long long *>(sm + Smem::DST);
    const uint32_t barA = smem_u32(sm + Smem::BAR), barO = barA + 8;
    uint32_t *s_slot = reinterpret_cast<uint32_t *>(sm + Smem::SLOT);
    int *s_abort = reinterpret_cast<int *>(sm + Smem::MISC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2;                       // warpgroup: column half of TMEM tiles
    const int trow = 32 * (warp & 3) + lane;        // this thread's TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *kk = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
    const __nv_bfloat16 *g = static_cast<const __nv_bfloat16 *>(a.g);
    const __nv_bfloat16 *qsb = static_cast<const __nv_bfloat16 *>(a.qs ? a.qs : a.q);
    const __nv_bfloat16 *ksb = static_cast<const __nv_bfloat16 *>(a.ks ? a.ks : a.k);

    // ---- segment ---------------------------------------------------------
    const int nshared = use_shared ? a.num_seqs * H : 0;
    const int P = N + use_shared;
    const bool is_shared = (int)blockIdx.x < nshared;
    int b, h, slot, len, base;
    if (is_shared) {
        b = blockIdx.x / H;
        h = blockIdx.x % H;
        slot = N;
        base = a.cu_seqlens[b];
        len = a.cu_seqlens[b + 1] - base;
    } else {
        const int s = blockIdx.x - nshared;
        slot = s % N;
        h = (s / N) % H;
        b = s / (N * H);
        base = a.seg_off[s];
        len = a.seg_off[s + 1] - base;
    }
    const __nv_bfloat16 *qsrc = is_shared ? qsb : q;
    const __nv_bfloat16 *ksrc = is_shared ? ksb : kk;
    const int64_t state_off = (((int64_t)b * H + h) * P + slot) * (int64_t)KC * DV;

    // ---- set-up: TMEM, barriers, zero padding atoms ----------------------
    if (warp == 0) tmem_alloc(smem_u32(s_slot), kTmemCols);
    if (tid == 0) {
        mbar_init(barA, 1);
        mbar_init(barO, 1);
        mbar_fence_init();
        *s_abort = 0;
    }
    if (KC < 128) {  // Kt is also the M = 128 operand of the state pass: its second atom stays 0
        for (int x = tid; x < kC * 8; x += kThreads) {
            const int r = x / 8, chunk = x % 8;
            *reinterpret_cast<uint4 *>(sK + (r >> 3) * 2048 + 1024 + (r & 7) * 128 + chunk * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_slot;
    const uint32_t tA = tmem + lane_base + kTmemA, tO = tmem + lane_base + kTmemO;
    const uint32_t tS = tmem + lane_base + kTmemS;

    // initial state -> TMEM (rows = key index = TMEM lane, fp32 columns)
    constexpr int kHalf = DV / 2;  // columns per warpgroup
    if (trow < KC) {
#pragma unroll
        for (int cb = 0; cb < kHalf; cb += 32) {
            uint32_t r[32];
            const int col0 = wg * kHalf + cb;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                r[i] = a.init ? __float_as_uint(a.init[state_off + (int64_t)trow * DV + col0 + i]) : 0u;
            tmem_st32(tS + col0, r);
        }
    }
    tmem_wait_st();
    float p_pending = 1.f;  // S_true[trow] = p_pending * S_stored[trow]

    const int nchunks = (len + kC - 1) / kC;
    for (int ch = 0; ch < nchunks; ++ch) {
        const uint32_t parity = ch & 1;
        // ---- row metadata --------------------------------------------------
        if (tid < kC) {
            const int n = ch * kC + tid;
            int t = -1;
            float e = 0.f;
            long long dst = -1;
            if (n < len) {
                if (is_shared) {
                    t = base + n;
                    e = 1.f;
                    dst = ((long long)t * H + h) * DV;
                } else {
                    const int rec = a.perm_rec[base + n];
                    t = rec / topk;
                    const int jj = rec - t * topk;
                    e = a.topk_w[((int64_t)t * H + h) * topk + jj];
                    dst = (((long long)t * H + h) * topk + jj) * DV;
                }
            }
            s_tok[tid] = t;
            s_e[tid] = e;
            s_dst[tid] = dst;
        }
        fence_before();
        __syncthreads();
        fence_after();

        // ---- transform: G cumsum, Qt, Kt (thread: 8 columns x RPT rows) ----
        constexpr int CG = KC / 8;              // column groups
        constexpr int NRB = kThreads / CG;      // row blocks
        constexpr int RPT = kC / NRB;           // rows per thread
        const int cg = tid % CG, rb = tid / CG;
        const int col0 = cg * 8;
        float G[RPT][8];
        {
            float run[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = rb * RPT + i;
                const int t = s_tok[r];
                if (t >= 0) {
                    float f[8];
                    unpack8(__ldg(reinterpret_cast<const uint4 *>(g + ((int64_t)t * H + h) * KC + col0)), f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) run[j] += f[j] * kLog2e;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) G[i][j] = run[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) s_tot[rb * 128 + col0 + j] = run[j];
        }
        __syncthreads();
        // per-column exclusive scan over row blocks; midpoint and last values
        if (tid < KC) {
            float acc = 0.f, gmid = 0.f;
            for (int r2 = 0; r2 < NRB; ++r2) {
                const float x = s_tot[r2 * 128 + tid];
                s_tot[r2 * 128 + tid] = acc;
                acc += x;
                if ((r2 + 1) * RPT - 1 == kMid) gmid = acc;
            }
            s_fmid[tid] = exp2f(gmid);
            s_beta[tid] = exp2f(acc - gmid);
            s_tot[32 * 128 + tid] = gmid;
        }
        __syncthreads();
        {
            float off[8], gm[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                off[j] = s_tot[rb * 128 + col0 + j];
                gm[j] = s_tot[32 * 128 + col0 + j];
            }
            bool range_bad = false;
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = rb * RPT + i;
                const int t = s_tok[r];
                uint4 qo = make_uint4(0, 0, 0, 0), ko = make_uint4(0, 0, 0, 0);
                if (t >= 0) {
                    const int64_t rowoff = ((int64_t)t * H + h) * KC + col0;
                    float fq[8], fk[8];
                    unpack8(__ldg(reinterpret_cast<const uint4 *>(qsrc + rowoff)), fq);
                    unpack8(__ldg(reinterpret_cast<const uint4 *>(ksrc + rowoff)), fk);
                    const float e = s_e[r];
                    const float eq = e * scale;
                    float qt[8], kt[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float dlt = G[i][j] + off[j] - gm[j];
                        range_bad |= fabsf(dlt) > kGateRangeLog2;
                        qt[j] = eq * fq[j] * exp2f(dlt);
                        kt[j] = e * fk[j] * exp2f(-dlt);
                    }
                    qo = make_uint4(pack_bf16x2(qt[0], qt[1]), pack_bf16x2(qt[2], qt[3]),
                                    pack_bf16x2(qt[4], qt[5]), pack_bf16x2(qt[6], qt[7]));
                    ko = make_uint4(pack_bf16x2(kt[0], kt[1]), pack_bf16x2(kt[2], kt[3]),
                                    pack_bf16x2(kt[4], kt[5]), pack_bf16x2(kt[6], kt[7]));
                }
                st_tile8(sQ, r, col0, qo);
                st_tile8(sK, r, col0, ko);
            }
            if (range_bad) atomicOr(a.flags, SSE_DEVICE_GATE_RANGE);
        }
        // V rows (raw bf16): thread covers 8 columns x VRPT rows
        {
            constexpr int VCG = DV / 8, VNRB = kThreads / VCG, VRPT = kC / VNRB;
            const int vcg = tid % VCG, vrb = tid / VCG;
#pragma unroll
            for (int i = 0; i < VRPT; ++i) {
                const int r = vrb * VRPT + i;
                const int t = s_tok[r];
                uint4 u = make_uint4(0, 0, 0, 0);
                if (t >= 0) u = __ldg(reinterpret_cast<const uint4 *>(v + ((int64_t)t * H + h) * DV + vcg * 8));
                st_tile8(sV, r, vcg * 8, u);
            }
        }
        // ---- state rows: S_stored *= exp(G_m) * p, bf16 copy -> sS ----------
        if (trow < KC) {
            const float f = s_fmid[trow] * p_pending;
#pragma unroll
            for (int cb = 0; cb < kHalf; cb += 32) {
                const int c0 = wg * kHalf + cb;
                uint32_t r[32];
                tmem_ld32(tS + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                tmem_st32(tS + c0, r);
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 u = make_uint4(
                        pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                        pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                        pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                        pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                    st_tile8(sS, trow, c0 + i, u);
                }
            }
            tmem_wait_st();
            p_pending = s_beta[trow];
        }
        fence_proxy_async();
        fence_before();
        __syncthreads();

        // ---- MMAs: A = Qt Kt^T; S += Kt^T V; O = Qt S' ------------------------
        if (tid == 0) {
            fence_after();
            const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV), s0 = smem_u32(sS);
            constexpr uint32_t idA = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idS = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t idO1 = idesc_bf16(128, DV, 0, 1);
#pragma unroll
            for (int k16 = 0; k16 < KC; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                mma_bf16(tmem + kTmemA, desc_sw128(q0 + ko, 16, 2048), desc_sw128(k0 + ko, 16, 2048), idA,
                         k16 > 0);
            }
            commit(barA);
#pragma unroll
            for (int k16 = 0; k16 < kC; k16 += 16) {
                const uint32_t ro = (k16 / 8) * 2048;
                mma_bf16(tmem + kTmemS, desc_sw128(k0 + ro, 1024, 2048), desc_sw128(v0 + ro, 1024, 2048), idS,
                         1);
            }
#pragma unroll
            for (int k16 = 0; k16 < KC; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                mma_bf16(tmem + kTmemO, desc_sw128(q0 + ko, 16, 2048),
                         desc_sw128(s0 + (k16 / 8) * 2048, 1024, 2048), idO1, k16 > 0);
            }
        }
        __syncwarp();

        // ---- P = mask(A) (bf16) ------------------------------------------------
        bool ok = mbar_wait_bounded(barA, parity, kWaitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(a.flags, SSE_DEVICE_TIMEOUT);
            break;
        }
        fence_after();
#pragma unroll
        for (int cb = 0; cb < 64; cb += 32) {
            const int c0 = wg * 64 + cb;
            uint32_t r[32];
            tmem_ld32(tA + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = (c0 + i + j <= trow) ? __uint_as_float(r[i + j]) : 0.f;
                st_tile8(sP, trow, c0 + i,
                         make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                    pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7])));
            }
        }
        fence_proxy_async();
        fence_before();
        __syncthreads();

        // ---- O += P V ------------------------------------------------------------
        if (tid == 0) {
            fence_after();
            const uint32_t p0 = smem_u32(sP), v0 = smem_u32(sV);
            constexpr uint32_t idO2 = idesc_bf16(128, DV, 0, 1);
#pragma unroll
            for (int k16 = 0; k16 < kC; k16 += 16) {
                const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                mma_bf16(tmem + kTmemO, desc_sw128(p0 + ko, 16, 2048),
                         desc_sw128(v0 + (k16 / 8) * 2048, 1024, 2048), idO2, 1);
            }
            commit(barO);
        }
        __syncwarp();
        ok = mbar_wait_bounded(barO, parity, kWaitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(a.flags, SSE_DEVICE_TIMEOUT);
            break;
        }
        fence_after();

        // ---- O rows -> fp32 partials ------------------------------------------
        {
            const long long dst = s_dst[trow];
            float *outp = is_shared ? a.part_shared : a.part_routed;
#pragma unroll
            for (int cb = 0; cb < kHalf; cb += 32) {
                const int c0 = wg * kHalf + cb;
                uint32_t r[32];
                tmem_ld32(tO + c0, r);
                tmem_wait_ld();
                if (dst >= 0) {
                    float4 *o4 = reinterpret_cast<float4 *>(outp + dst + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        o4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            }
        }
        fence_before();
        __syncthreads();
        fence_after();
    }

    // ---- final state = p * S_stored --------------------------------------------
    if (a.final_state && trow < KC) {
#pragma unroll
        for (int cb = 0; cb < kHalf; cb += 32) {
            const int c0 = wg * kHalf + cb;
            uint32_t r[32];
            tmem_ld32(tS + c0, r);
            tmem_wait_ld();
            float4 *o4 = reinterpret_cast<float4 *>(a.final_state + state_off + (int64_t)trow * DV + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                o4[i] = make_float4(__uint_as_float(r[4 * i]) * p_pending, __uint_as_float(r[4 * i + 1]) * p_pending,
                                    __uint_as_float(r[4 * i + 2]) * p_pending,
                                    __uint_as_float(r[4 * i + 3]) * p_pending);
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int KC, int DV>
cudaError_t launch_t(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    static bool attr_set = false;  // benign race: the attribute value is the same for every caller
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunked_segment_kernel<KC, DV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t nseg = (int64_t)a.num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    if (nseg == 0) return cudaSuccess;
    chunked_segment_kernel<KC, DV><<<(unsigned)nseg, kThreads, kSmemBytes, stream>>>(
        a, cfg.num_heads, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale);
    return cudaGetLastError();
}

}  // namespace

bool chunked_supported(const sse_config_t &cfg) {
    const bool c_ok = cfg.key_dim == 64 || cfg.key_dim == 128;
    const bool d_ok = cfg.value_dim == 64 || cfg.value_dim == 128;
    return cfg.dtype == SSE_BF16 && c_ok && d_ok;
}

size_t chunked_extra_workspace(const sse_config_t &, int64_t, int32_t) { return 0; }

cudaError_t launch_forward_chunked(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream,
                                   int *launches) {
    cudaError_t e;
    if (cfg.key_dim == 128 && cfg.value_dim == 128) e = launch_t<128, 128>(cfg, a, stream);
    else if (cfg.key_dim == 128 && cfg.value_dim == 64) e = launch_t<128, 64>(cfg, a, stream);
    else if (cfg.key_dim == 64 && cfg.value_dim == 128) e = launch_t<64, 128>(cfg, a, stream);
    else if (cfg.key_dim == 64 && cfg.value_dim == 64) e = launch_t<64, 64>(cfg, a, stream);
    else return cudaErrorInvalidValue;
    *launches += 1;
    if (e != cudaSuccess) return e;
    e = launch_combine(cfg, a, stream);
    *launches += 1;
    return e;
}

}  // namespace sse
