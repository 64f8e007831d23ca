// front_end.cu -- tensor-core (tcgen05 + TMEM, TMA-fed) front end of the SSE
// layer.
//
// "Scaling Linear Attention with Sparse State Expansion", eqs. 9-10, per head:
// q = x W_q, k = softmax(x W_k) over the c keys, v = x W_v and the router
// logits x W_e; GLA's diagonal gate as the log-gate g = logsigmoid(x W_g) / tau;
// and (section 2.5) the shared partition's q and k through a rank-64 LoRA of
// W_q and W_k: q^s = x W_q + (x A_q) B_q, k^s = softmax(x W_k + (x A_k) B_k).
// Weights use the [out_features, in_features] layout (y = x W^T), so every
// operand is K-major.
//
// One persistent kernel computes output tiles of 128 tokens x one projection
// block, K = D in steps of 64 (one 128-byte swizzle atom).  Blocks: one
// head's [q | k] (N = 2c) or [v | g] (N = d + c), and all heads' router
// logits.  The wide blocks halve the x tiles read per output and the
// shared-memory operand traffic per flop (an N = 128 MMA reads as many
// operand bytes per flop as the shared memory delivers).
//   warp 0 (lane 0): TMA loads of each step's x tile and weight tile into a
//       four-stage ring;
//   warp 1 (lane 0): the tcgen05 MMAs (M = 128, N = block width, K = 16) into
//       one of two TMEM accumulators; once the epilogue has read q and k of a
//       [q | k] tile, two more K steps add the LoRA terms (x A_q) B_q and
//       (x A_k) B_k onto the same columns (issued half way through the next
//       tile's mainloop), and the epilogue reads q^s and k^s;
//   warps 2-5 (one TMEM lane = one token each): the block's epilogue
//       (identity, key softmax, log-sigmoid gate) from TMEM to bf16 outputs,
//       while the MMAs of the next tile fill the other accumulator.
// x A (both LoRA first factors, [T, 128]) comes from a first launch of the
// same kernel over two 64-wide blocks.  All waits are bounded (a timeout sets
// SSE_DEVICE_TIMEOUT and the roles stop).
#include <algorithm>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "sse_internal.cuh"
#include "umma.cuh"

namespace sse {
namespace {

using namespace umma;

constexpr int kRows = 128;                 // tokens per tile (TMEM lanes)
constexpr int kKStep = 64;                 // K elements per stage (one swizzle atom)
constexpr int kStages = 4;
constexpr uint32_t kATile = kRows * 128;   // 16 KB
constexpr uint32_t kBTileMax = 256 * 128;  // 32 KB (N up to 256)
constexpr uint32_t kStageBytes = kATile + kBTileMax;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 512;        // two accumulators of 256 columns
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

enum { kBarFull = 0, kBarEmpty = kStages, kBarAccF = 2 * kStages, kBarAccE = 2 * kStages + 2,
       kBarAccM = 2 * kStages + 4,  // first read-out of a [q | k] tile done (before its LoRA steps)
       kNumBars = 2 * kStages + 6 };
constexpr uint32_t kSmemBar = kStages * kStageBytes;
constexpr size_t kSmemBytes = kSmemBar + 8 * kNumBars + 16 + 1024;

// Block kinds.  Phase 1: one head's [q | k] or [v | g], or all heads' logits;
// phase 0: the two LoRA first factors x A_q, x A_k.
enum Kind { kQK = 0, kVG, kE, kXAq, kXAk };

struct FeArgs {
    int32_t T, D, H, c, d, Np, has_lora, phase;
    float gate_inv_tau;
    __nv_bfloat16 *q, *k, *v, *g, *logits, *qs, *ks, *xa;
    int32_t *flags;
};

struct FeMaps {
    CUtensorMap x, xa, wq, wk, wv, wg, we, aq, ak, bq, bk;
};

// n = n1 + n2: a pair block's B tile stacks n1 rows of its first weight and
// n2 rows of its second.
struct Tile {
    int row0, kind, h, n, n1;
};

// phase 1: [q|k]_0..[q|k]_{H-1}, [v|g]_0.., logits (2H + 1 blocks)
__device__ __forceinline__ int num_col_blocks(const FeArgs &a) { return a.phase == 0 ? 2 : 2 * a.H + 1; }

__device__ __forceinline__ Tile decode_tile(const FeArgs &a, int tile) {
    const int ncol = num_col_blocks(a);
    Tile t;
    t.row0 = (tile / ncol) * kRows;
    const int cb = tile % ncol;
    t.h = 0;
    if (a.phase == 0) {
        t.kind = kXAq + cb;
        t.n = t.n1 = 64;
    } else if (cb == ncol - 1) {
        t.kind = kE;
        t.n = t.n1 = a.H * a.Np;
    } else {
        t.kind = cb < a.H ? kQK : kVG;
        t.h = cb % a.H;
        t.n1 = t.kind == kVG ? a.d : a.c;
        t.n = t.n1 + a.c;
    }
    return t;
}

__device__ __forceinline__ bool has_lora_step(const FeArgs &a, const Tile &t) {
    return a.has_lora && t.kind == kQK;
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(mbar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(mbar), "r"(bytes) : "memory");
}
// TMA load of one box of a 2-D tensor map (inner coordinate x, row y) into
// shared memory, completion counted in bytes on mbar.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap *map, uint32_t sdst, uint32_t mbar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(sdst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// logsigmoid(y) = min(y, 0) - log(1 + exp(-|y|))
__device__ __forceinline__ float log_sigmoid(float y) { return fminf(y, 0.f) - log1pf(__expf(-fabsf(y))); }

// Writes the first `cnt` (16 or 32) of 32 values of this lane's row as bf16
// (16-byte stores).
__device__ __forceinline__ void store32(__nv_bfloat16 *dst, const float (&f)[32], int cnt = 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 8)
        if (i < cnt) *reinterpret_cast<uint4 *>(dst + i) =
            make_uint4(pack_bf16x2(f[i], f[i + 1]), pack_bf16x2(f[i + 2], f[i + 3]),
                       pack_bf16x2(f[i + 4], f[i + 5]), pack_bf16x2(f[i + 6], f[i + 7]));
}

// 32 accumulator columns of this lane.
__device__ __forceinline__ void load_acc(uint32_t tacc, int c0, float (&f)[32]) {
    uint32_t r[32];
    tmem_ld32(tacc + c0, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(r[i]);
}

// Plain block: y -> bf16 (optionally the gate transform).  n is a multiple of
// 16 (the router block can end half way through a 32-column load).
__device__ __forceinline__ void epi_plain(uint32_t tacc, int n, bool gate, float inv_tau, __nv_bfloat16 *dst) {
    for (int c0 = 0; c0 < n; c0 += 32) {
        float f[32];
        load_acc(tacc, c0, f);
        if (gate) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = log_sigmoid(f[i]) * inv_tau;
        }
        if (dst) store32(dst + c0, f, min(32, n - c0));
    }
}

// Key block: softmax over the row's n columns -> bf16.
__device__ __forceinline__ void epi_softmax(uint32_t tacc, int n, __nv_bfloat16 *dst) {
    float m = -INFINITY;
    for (int c0 = 0; c0 < n; c0 += 32) {
        float f[32];
        load_acc(tacc, c0, f);
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, f[i]);
    }
    const float mb = m * kLog2e;
    float s = 0.f;
    for (int c0 = 0; c0 < n; c0 += 32) {
        float f[32];
        load_acc(tacc, c0, f);
#pragma unroll
        for (int i = 0; i < 32; ++i) s += ex2(fmaf(f[i], kLog2e, -mb));
    }
    const float inv = 1.f / s;
    for (int c0 = 0; c0 < n; c0 += 32) {
        float f[32];
        load_acc(tacc, c0, f);
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = ex2(fmaf(f[i], kLog2e, -mb)) * inv;
        if (dst) store32(dst + c0, f);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
front_end_kernel(FeArgs a, const __grid_constant__ FeMaps maps, int32_t num_tiles) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t bar0 = smem_u32(sm + kSmemBar);
    auto bar = [&](int i) { return bar0 + 8u * i; };
    uint32_t *s_slot = reinterpret_cast<uint32_t *>(sm + kSmemBar + 8 * kNumBars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) tmem_alloc(smem_u32(s_slot), kTmemCols);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarFull + s), 1);
            mbar_init(bar(kBarEmpty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kBarAccF + b), 1);
            mbar_init(bar(kBarAccE + b), 128);
            mbar_init(bar(kBarAccM + b), 128);
        }
        mbar_fence_init();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_slot;
    const int nk_main = a.D / kKStep;
    bool failed = false;

    // The LoRA steps of a [q | k] tile (two K steps of 64: (x A_q) B_q onto the
    // q columns, (x A_k) B_k onto the k columns) run after the epilogue has
    // read q and k, half way through the next tile's mainloop (or right after
    // the tile when it is this CTA's last).  Producer and MMA warp walk the same
    // stage sequence.
    const int lora_at = nk_main / 2;

    if (warp == 0) {
        // ---- TMA producer ----------------------------------------------------
        uint32_t it = 0;
        if (lane == 0) {
            auto next_stage = [&](uint32_t bytes) -> int {  // -1 on timeout
                const int s = it % kStages;
                if (it >= kStages && !mbar_wait_bounded(bar(kBarEmpty + s), ((it / kStages) - 1) & 1, kWaitNs))
                    return -1;
                mbar_arrive_expect_tx(bar(kBarFull + s), bytes);
                ++it;
                return s;
            };
            auto emit_lora = [&](const Tile &t) -> bool {
                for (int half = 0; half < 2; ++half) {
                    const int s = next_stage(kATile + (uint32_t)a.c * 128u);
                    if (s < 0) return false;
                    const uint32_t sa = smem_u32(sm + s * kStageBytes), sb = sa + kATile;
                    tma_load_2d(&maps.xa, sa, bar(kBarFull + s), half * 64, t.row0);
                    tma_load_2d(half ? &maps.bk : &maps.bq, sb, bar(kBarFull + s), 0, t.h * a.c);
                }
                return true;
            };
            bool pend = false;
            Tile tp{};
            for (int tile = blockIdx.x; tile < num_tiles && !failed; tile += gridDim.x) {
                const Tile t = decode_tile(a, tile);
                // first (and, for pair blocks, second) weight of the block, with the
                // row of its first output
                const CUtensorMap *w1 = t.kind == kQK ? &maps.wq : t.kind == kVG ? &maps.wv
                                      : t.kind == kE ? &maps.we : t.kind == kXAq ? &maps.aq : &maps.ak;
                const CUtensorMap *w2 = t.kind == kQK ? &maps.wk : t.kind == kVG ? &maps.wg : nullptr;
                const int r1 = t.kind == kVG ? t.h * a.d : t.h * a.c, r2 = t.h * a.c;
                for (int ks = 0; ks < nk_main; ++ks) {
                    if (pend && ks == lora_at) {
                        if (!emit_lora(tp)) { failed = true; break; }
                        pend = false;
                    }
                    const int s = next_stage(kATile + (uint32_t)t.n * 128u);
                    if (s < 0) { failed = true; break; }
                    const uint32_t sa = smem_u32(sm + s * kStageBytes), sb = sa + kATile;
                    tma_load_2d(&maps.x, sa, bar(kBarFull + s), ks * kKStep, t.row0);
                    tma_load_2d(w1, sb, bar(kBarFull + s), ks * kKStep, r1);
                    if (w2) tma_load_2d(w2, sb + (uint32_t)t.n1 * 128u, bar(kBarFull + s), ks * kKStep, r2);
                }
                if (has_lora_step(a, t)) {
                    pend = true;
                    tp = t;
                }
            }
            if (!failed && pend && !emit_lora(tp)) failed = true;
            // no copy may still be writing shared memory when the CTA exits
            for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
                if (!mbar_wait_bounded(bar(kBarFull + j % kStages), (j / kStages) & 1, kWaitNs)) failed = true;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue ----------------------------------------------------------
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            uint32_t mpar = 0;  // bit b: parity of the next first-read-out phase of accumulator b
            auto take_stage = [&](uint32_t &sa, uint32_t &sb) -> bool {
                const int s = it % kStages;
                if (!mbar_wait_bounded(bar(kBarFull + s), (it / kStages) & 1, kWaitNs)) return false;
                fence_after();
                sa = smem_u32(sm + s * kStageBytes);
                sb = sa + kATile;
                return true;
            };
            auto release_stage = [&]() { commit(bar(kBarEmpty + (it % kStages))); ++it; };
            // (x A) B onto the q and k columns of accumulator b, once its first
            // read-out is done; then the second "accumulator full".
            auto do_lora = [&](int b) -> bool {
                if (!mbar_wait_bounded(bar(kBarAccM + b), (mpar >> b) & 1, kWaitNs)) return false;
                mpar ^= 1u << b;
                fence_after();
                const uint32_t idl = idesc_bf16(kRows, a.c, 0, 0);
                for (int half = 0; half < 2; ++half) {
                    uint32_t sa, sb;
                    if (!take_stage(sa, sb)) return false;
#pragma unroll
                    for (int k16 = 0; k16 < kKStep; k16 += 16)
                        mma_bf16(tmem + (uint32_t)b * 256u + (uint32_t)(half * a.c), desc_sw128(sa + k16 * 2, 16, 1024),
                                 desc_sw128(sb + k16 * 2, 16, 1024), idl, 1);
                    release_stage();
                }
                commit(bar(kBarAccF + b));
                return true;
            };
            int pend_b = -1;
            for (int tile = blockIdx.x; tile < num_tiles && !failed; tile += gridDim.x, ++tc) {
                const Tile t = decode_tile(a, tile);
                const int b = tc & 1;
                if (tc >= 2 && !mbar_wait_bounded(bar(kBarAccE + b), ((tc >> 1) - 1) & 1, kWaitNs)) {
                    failed = true;
                    break;
                }
                fence_after();
                const uint32_t acc = tmem + (uint32_t)b * 256u;
                const uint32_t idesc = idesc_bf16(kRows, t.n, 0, 0);
                for (int ks = 0; ks < nk_main; ++ks) {
                    if (pend_b >= 0 && ks == lora_at) {
                        if (!do_lora(pend_b)) { failed = true; break; }
                        pend_b = -1;
                    }
                    uint32_t sa, sb;
                    if (!take_stage(sa, sb)) { failed = true; break; }
#pragma unroll
                    for (int k16 = 0; k16 < kKStep; k16 += 16)
                        mma_bf16(acc, desc_sw128(sa + k16 * 2, 16, 1024), desc_sw128(sb + k16 * 2, 16, 1024), idesc,
                                 (ks + k16) > 0);
                    release_stage();
                }
                if (failed) break;
                commit(bar(kBarAccF + b));
                if (has_lora_step(a, t)) pend_b = b;
            }
            if (!failed && pend_b >= 0 && !do_lora(pend_b)) failed = true;
        }
        __syncwarp();
    } else {
        // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 ---------------
        const int row = 32 * (warp & 3) + lane;
        const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t tc = 0;
        uint32_t fpar = 0;  // bit b: parity of the next "accumulator full" phase of accumulator b
        auto wait_full = [&](int b) -> bool {
            const bool ok = mbar_wait_bounded(bar(kBarAccF + b), (fpar >> b) & 1, kWaitNs);
            fpar ^= 1u << b;
            if (!__all_sync(0xffffffffu, ok)) return false;
            fence_after();
            return true;
        };
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
            const Tile t = decode_tile(a, tile);
            const int b = tc & 1;
            if (!wait_full(b)) {
                failed = true;
                break;
            }
            const uint32_t tacc = tmem + lb + (uint32_t)b * 256u;
            const int tok = t.row0 + row;
            const bool live = tok < a.T;
            const int64_t hc = (int64_t)a.H * a.c;
            switch (t.kind) {
            case kQK:  // columns [0, c): q; [c, 2c): the key logits
                epi_plain(tacc, a.c, false, 0.f, live ? a.q + tok * hc + t.h * a.c : nullptr);
                epi_softmax(tacc + a.c, a.c, live ? a.k + tok * hc + t.h * a.c : nullptr);
                if (has_lora_step(a, t)) {  // the same columns after the LoRA steps
                    fence_before();
                    mbar_arrive(bar(kBarAccM + b));
                    if (!wait_full(b)) {
                        failed = true;
                        break;
                    }
                    epi_plain(tacc, a.c, false, 0.f, live ? a.qs + tok * hc + t.h * a.c : nullptr);
                    epi_softmax(tacc + a.c, a.c, live ? a.ks + tok * hc + t.h * a.c : nullptr);
                }
                break;
            case kVG:  // columns [0, d): v; [d, d + c): the gate
                epi_plain(tacc, a.d, false, 0.f, live ? a.v + tok * (int64_t)a.H * a.d + t.h * a.d : nullptr);
                epi_plain(tacc + a.d, a.c, true, a.gate_inv_tau, live ? a.g + tok * hc + t.h * a.c : nullptr);
                break;
            case kE:
                epi_plain(tacc, t.n, false, 0.f, live ? a.logits + tok * (int64_t)t.n : nullptr);
                break;
            default:  // x A_q -> columns 0..63, x A_k -> 64..127
                epi_plain(tacc, t.n, false, 0.f,
                          live ? a.xa + tok * (int64_t)128 + (t.kind == kXAq ? 0 : 64) : nullptr);
                break;
            }
            if (failed) break;
            fence_before();
            mbar_arrive(bar(kBarAccE + b));
        }
    }
    if (failed) atomicOr(a.flags, SSE_DEVICE_TIMEOUT);
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A [rows, cols] bf16 row-major matrix, loaded in boxes of 64 columns x
// box_rows rows with the 128-byte swizzle (rows past the end read as zero).
bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *base, int64_t rows,
               int64_t cols, int box_rows) {
    memset(m, 0, sizeof *m);
    if (!base) return true;  // never read
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool front_end_supported(const sse_config_t &cfg, int32_t hidden) {
    const int hn = cfg.num_heads * cfg.num_partitions;
    return cfg.dtype == SSE_BF16 && (cfg.key_dim == 64 || cfg.key_dim == 128) &&
           (cfg.value_dim == 64 || cfg.value_dim == 128) && hidden >= 64 && hidden % 64 == 0 && hn % 16 == 0 &&
           hn <= 256;
}

cudaError_t launch_front_end(const sse_config_t &cfg, const FrontEndArgs &f, cudaStream_t stream, int *launches) {
    static bool attr_set = false;  // benign race: every caller sets the same value
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(front_end_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (f.T == 0) return cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const int H = cfg.num_heads, c = cfg.key_dim, d = cfg.value_dim, Np = cfg.num_partitions;
    const int64_t D = f.hidden, T = f.T;
    const bool lora = f.a_q != nullptr;
    FeMaps m;
    bool ok = encode_2d(enc, &m.x, f.x, T, D, kRows) && encode_2d(enc, &m.xa, lora ? f.xa : nullptr, T, 128, kRows) &&
              encode_2d(enc, &m.wq, f.w_q, (int64_t)H * c, D, c) && encode_2d(enc, &m.wk, f.w_k, (int64_t)H * c, D, c) &&
              encode_2d(enc, &m.wv, f.w_v, (int64_t)H * d, D, d) && encode_2d(enc, &m.wg, f.w_g, (int64_t)H * c, D, c) &&
              encode_2d(enc, &m.we, f.w_e, (int64_t)H * Np, D, H * Np) &&
              encode_2d(enc, &m.aq, f.a_q, 64, D, 64) && encode_2d(enc, &m.ak, f.a_k, 64, D, 64) &&
              encode_2d(enc, &m.bq, f.b_q, (int64_t)H * c, 64, c) && encode_2d(enc, &m.bk, f.b_k, (int64_t)H * c, 64, c);
    if (!ok) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    FeArgs a{};
    a.T = (int32_t)T;
    a.D = (int32_t)D;
    a.H = H;
    a.c = c;
    a.d = d;
    a.Np = Np;
    a.has_lora = lora ? 1 : 0;
    a.gate_inv_tau = f.gate_inv_tau;
    a.q = static_cast<__nv_bfloat16 *>(f.q);
    a.k = static_cast<__nv_bfloat16 *>(f.k);
    a.v = static_cast<__nv_bfloat16 *>(f.v);
    a.g = static_cast<__nv_bfloat16 *>(f.g);
    a.logits = static_cast<__nv_bfloat16 *>(f.logits);
    a.qs = static_cast<__nv_bfloat16 *>(f.q_shared);
    a.ks = static_cast<__nv_bfloat16 *>(f.k_shared);
    a.xa = static_cast<__nv_bfloat16 *>(f.xa);
    a.flags = f.flags;
    const int64_t row_tiles = (T + kRows - 1) / kRows;
    for (int phase = lora ? 0 : 1; phase <= 1; ++phase) {
        a.phase = phase;
        const int64_t tiles = row_tiles * (phase == 0 ? 2 : 2 * H + 1);
        const int grid = (int)std::min<int64_t>(tiles, sms);
        front_end_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, m, (int32_t)tiles);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    return cudaSuccess;
}

}  // namespace sse
