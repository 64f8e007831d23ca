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
//   Qt_r = q_r * exp(G_r - G_m)                  Kt_s = e_s k_s * exp(G_m - G_s)
//   A    = Qt Kt^T, causally masked (s <= r) -> P (bf16)
//   O_r  = e_r scale [Qt (exp(G_m) * S) + P V]_r     (inter- + intra-chunk)
//   S'   = exp(G_last) * S + exp(G_last - G_m) * Kt^T V   (state pass)
//
// Every factor exp(+-(G_r - G_m)) is bounded by exp(|G| over half a chunk),
// which is why the chunk is split at its midpoint.  The state S (c x d,
// fp32) lives in TMEM for the whole segment as S = p * S_stored with a
// per-row pending scale p: each chunk rescales S_stored by exp(G_m) * p in
// place (also producing the bf16 copy used by Qt S), lets the tensor core
// accumulate Kt^T V into it, and sets p = exp(G_last - G_m).
//
// Persistent CTAs (one per SM) take segments from an atomic queue (shared
// segments first: they are the longest).  Inside a CTA three warp roles run a
// pipeline synchronised by mbarriers:
//   loader (4 warps): warp 0 claims the work items, hands each segment to the
//       other roles and writes every chunk's row metadata (token, router
//       weight) into a ring a few chunks ahead; warp 1 has the TMA engine
//       gather each chunk's V rows into a double buffer (tile::gather4, four
//       token rows per copy, 128B swizzle, straight into the operand layout);
//   transform (8 warps): load the chunk's raw q and k rows between the row
//       sums of its first pass over g, and the next chunk's g rows inside the
//       decay pass (into the registers each row has just released); scan g
//       (which releases the epilogue's state-row pass); build Qt and Kt
//       (128B-swizzled, see umma.cuh);
//   epilogue (4 warps, one TMEM lane each): rescale the state rows and
//       write S'; turn A into the masked bf16 P; write O (already e-weighted)
//       as bf16 partial rows; final state at the end of the segment.  Lane 0
//       of warp 0 also issues the tensor-core work of each chunk at the
//       points of its loop where the operands become ready:
//       A = Qt Kt^T; S += Kt^T V; O = Qt S' (after the state rows), then
//       O += P V (after P).
// All waits are bounded: a timeout sets SSE_DEVICE_TIMEOUT in the flags word
// and the CTA stops after releasing its TMEM.
#include <algorithm>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "sse_internal.cuh"
#include "f32x2.cuh"
#include "umma.cuh"

namespace sse {
namespace {

using namespace umma;

constexpr int kC = kChunkRows;   // chunk rows (128)
constexpr int kMid = kC / 2 - 1; // midpoint row of the decay split
constexpr int kEpiWarps = 4, kTrfWarps = 8, kLdrWarps = 4;
constexpr int kThreads = 32 * (kEpiWarps + kTrfWarps + kLdrWarps);  // 512: 4 warps per SM sub-partition
constexpr int kTrfThreads = 32 * kTrfWarps;
// Registers per thread: at launch (65536 / 512) and after the split between
// the warpgroups (setmaxnreg).
constexpr int kRegsLaunch = 128, kRegsEpi = 120, kRegsTrf = 176, kRegsLdr = 40;
static_assert(32 * (kEpiWarps * kRegsEpi + kTrfWarps * kRegsTrf + kLdrWarps * kRegsLdr) == kThreads * kRegsLaunch,
              "register split must use exactly the launch allocation");
#ifdef SSE_FAULT_INJECT
// Checked build (libsse_checked.so, for the failure-detection test only):
// every bounded wait gives up after 50 ms, and g_fault_mode = 1 makes CTA 0's
// transform warps withhold their "Qt / Kt written" arrival for the first
// chunk, so that the waits on it run out and the kernel takes its abort path
// (SSE_DEVICE_TIMEOUT, roles stop together, TMEM freed).  Nothing faults or
// hangs: every wait in the kernel is bounded.
__device__ int g_fault_mode = 0;
constexpr uint64_t kWaitNs = 50000000ull;
#else
constexpr uint64_t kWaitNs = 2000000000ull;
#endif
constexpr float kLog2e = 1.4426950408889634f;
// Largest |G_r - G_m| (summed log-gate over a half chunk, per key row) the
// factorised form takes.  Every factor exp(+-(G_r - G_m)) then stays within
// e^64: a bf16 operand that underflows (below ~1e-38) is multiplied by at most
// e^64 (~6e27) in any product, so what rounding loses there stays below
// ~1e-10 of |q| |k| |v| -- far under bf16's own rounding.  A chunk past it is
// not evaluated in factorised form: its whole segment goes to the redo list
// and is recomputed token by token (segment_redo_kernel).
constexpr float kGateRange = 64.f;

constexpr uint32_t kTile = 128 * 256;   // one 128 x 128 bf16 tile: 32 KB
// Row metadata ring (global chunk g in stage g % kMetaStages): written by the
// loader, read by the gather warps, the transform and, last, by the epilogue
// when it writes the chunk's output; the loader reuses a stage after that
// (kBarMF), so it runs up to about three chunks ahead of the transform.
constexpr int kMetaStages = 5;

// Segment hand-off ring: the loader posts each work item's description (or
// the end of the work) for the transform and epilogue warps, so that the roles
// move between segments independently.
constexpr int kSegSlots = 4;

enum Bar {
    kBarT = 0, kBarSc0, kBarSc1, kBarS, kBarA, kBarQK, kBarP, kBarO, kBarOf0, kBarOf1, kBarV0, kBarV1,
    kBarVL0, kBarVL1,                  // V rows of a chunk landed in V0 / V1 (TMA)
    kBarMR,                            // kMetaStages "row metadata written" barriers
    kBarMF = kBarMR + kMetaStages,     // kMetaStages "row metadata no longer needed" barriers
    kBarSegF = kBarMF + kMetaStages,   // kSegSlots "descriptor posted" barriers
    kBarSegE = kBarSegF + kSegSlots,   // kSegSlots "descriptor consumed" barriers
    kNumBars = kBarSegE + kSegSlots
};

// Shared-memory layout (offsets from a 1024-aligned base).
struct Smem {
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t K = Q + kTile;
    static constexpr uint32_t V0 = K + kTile;
    static constexpr uint32_t V1 = V0 + kTile;
    static constexpr uint32_t P = V1 + kTile;
    // the S' tile doubles as the output staging tile (see write_out)
    static constexpr uint32_t S = P + kTile;
    static constexpr uint32_t TOT = S + kTile;             // [33][128] f32 block prefixes; row 32: G_m
    static constexpr uint32_t SCALE = TOT + 33 * 128 * 4;  // [2 stages][2][128] f32: exp(G_m), exp(G_last-G_m)
    // [kMetaStages] x {tok[128], e[128], header {stop, h, shared, -}}
    static constexpr uint32_t META = SCALE + 2 * 2 * 128 * 4;
    static constexpr uint32_t META_STAGE = 128 * (4 + 4) + 16;
    static constexpr uint32_t SEGQ = META + kMetaStages * META_STAGE;  // [kSegSlots][8] int
    static constexpr uint32_t BAR = SEGQ + kSegSlots * 32;
    static constexpr uint32_t MISC = BAR + 8 * kNumBars;   // TMEM slot, work item
    static constexpr uint32_t END = MISC + 16;
};
constexpr size_t kSmemBytes = Smem::END + 1024;  // + alignment slack

// TMEM columns: A (Qt Kt^T), two O buffers (chunk parity), the state S.
constexpr uint32_t kTmemA = 0, kTmemO0 = 128, kTmemS = 256, kTmemO1 = 384, kTmemCols = 512;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Product of two bf16x2 words (round to nearest).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
    __nv_bfloat162 z = __hmul2(x, y);
    return *reinterpret_cast<uint32_t *>(&z);
}

__device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t tile_off(int row, int col) { return sw128_offset(row, col, 2); }

// 2^x with the SFU instruction (relative error ~2^-22, flushes denormals);
// its operands are rounded to bf16 right after.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int R> __device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(R));
}
template <int R> __device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(R));
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(mbar) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads,
// so that every participant takes the same branch afterwards.
__device__ __forceinline__ bool named_sync_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(count) : "memory");
    return r != 0;
}
// 16-byte read-only global load that does not keep its line in L1 (each row
// piece is read once per CTA).
__device__ __forceinline__ uint4 ldg_stream(const void *gptr) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(gptr));
    return r;
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Prefetch into L2 of the 128-byte lines of `bytes` of global memory starting
// at a 128-byte boundary (plain per-thread prefetches: no completion to wait
// for, and nothing queued on the TMA engine).
__device__ __forceinline__ void prefetch_l2(const void *gptr, uint32_t bytes) {
    for (uint32_t o = 0; o < bytes; o += 128)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(static_cast<const char *>(gptr) + o));
}
// Tensor (TMA) store of one box of a 2-D tensor map from shared memory; the
// box's inner coordinate x and row coordinate y.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t ssrc, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(ssrc), "r"(x), "r"(y) : "memory");
}
// Waits until this thread's bulk copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Arrive on an mbarrier and raise the bytes its phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(mbar), "r"(bytes) : "memory");
}
// TMA gather of four rows (r0..r3) x one box of columns starting at x of a 2-D
// tensor map whose box is one row high; the rows land one after another at
// sdst (the map's swizzle applied), completion counted on mbar in bytes.
__device__ __forceinline__ void tma_gather4(const CUtensorMap *map, uint32_t sdst, uint32_t mbar, int x, int r0,
                                            int r1, int r2, int r3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        :: "r"(sdst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(mbar)
        : "memory");
}


struct Segment {
    int b, h, slot, base, len;
    bool shared;
};

// Work items: the shared segments first (the longest, so the persistent CTAs
// start them early), then the routed segments s = (b * H + h) * N + i: the
// grouped records of partition i, or (masking schedule) the whole sequence b.
template <bool MASKED>
__device__ __forceinline__ Segment decode_segment(const ForwardArgs &a, int item, int H, int N,
                                                  int use_shared) {
    Segment s;
    const int nshared = use_shared ? a.num_seqs * H : 0;
    s.shared = item < nshared;
    if (s.shared) {
        s.b = item / H;
        s.h = item % H;
        s.slot = N;
        s.base = a.cu_seqlens[s.b];
        s.len = a.cu_seqlens[s.b + 1] - s.base;
    } else {
        const int r = item - nshared;
        s.slot = r % N;
        s.h = (r / N) % H;
        s.b = r / (N * H);
        if (MASKED) {
            s.base = a.cu_seqlens[s.b];
            s.len = a.cu_seqlens[s.b + 1] - s.base;
        } else {
            // routing outputs: L2 loads (see the routing kernels' dependent launches)
            s.base = __ldcg(a.seg_off + r);
            s.len = __ldcg(a.seg_off + r + 1) - s.base;
        }
    }
    return s;
}

// Queue position -> work item.  With the shared partition on, the (sequence,
// head) pairs go in waves of kWavePairs: a wave's shared segments first (the
// longest items, started early), then its routed segments pair by pair, so
// that more of the k + 1 reads of a token row meet in L2.  Measured on GB300
// (main kernel, layer workload 8 x 4096 tokens H16 N8 / varlen 16 sequences
// H16 N16, one box): plain order 0.430 / 3.19 ms; waves of 16 pairs
// 0.466 / 3.50; 32: 0.429 / 3.46; 48: 0.429 / 3.55; 64: 0.418 / 3.18.
constexpr int kWavePairs = 64;
__device__ __forceinline__ int queue_item(int qpos, int npairs, int N, int use_shared) {
    if (!use_shared) return qpos;
    const int per_wave = kWavePairs * (N + 1);
    const int w = qpos / per_wave, r = qpos - w * per_wave;
    const int p0 = w * kWavePairs;
    const int wc = min(kWavePairs, npairs - p0);  // pairs in this wave (the last one may be short)
    if (r < wc) return p0 + r;                     // shared segment of pair p0 + r
    const int rr = r - wc;
    return npairs + (p0 + rr / N) * N + rr % N;    // routed segment (pair, partition)
}

// Row metadata of row idx of a work item: token index and router weight.
struct RowMeta { int t; float e; };
template <bool MASKED>
__device__ __forceinline__ RowMeta row_meta(const ForwardArgs &a, const Segment &seg, int idx, int H, int topk) {
    RowMeta m{-1, 0.f};
    if (idx < seg.len) {
        if (seg.shared) {
            m.t = seg.base + idx;
            m.e = 1.f;
        } else if (MASKED) {
            // every token of the sequence; -1 marks the ones that did not select
            // this partition (no write, no decay, no read)
            m.t = seg.base + idx;
            m.e = -1.f;
            const int64_t o = ((int64_t)m.t * H + seg.h) * topk;
            for (int j = 0; j < topk; ++j)
                if (__ldcg(a.topk_idx + o + j) == seg.slot) m.e = __ldcg(a.topk_w + o + j);
        } else {
            m.t = __ldcg(a.perm_rec + seg.base + idx) / topk;
            m.e = __ldcg(a.perm_e + seg.base + idx);
        }
    }
    return m;
}

// Tensor map of v as a 2-D [T * H, d] bf16 array, boxes of 64 columns x 1 row,
// 128-byte swizzle (the TMA gathers of the loader).
struct RowMaps {
    CUtensorMap v;
};

template <int KC, int DV, bool MASKED>
__global__ void __launch_bounds__(kThreads, 1)
chunked_forward_kernel(ForwardArgs a, const __grid_constant__ CUtensorMap part_map,
                       const __grid_constant__ RowMaps maps, int32_t H, int32_t N, int32_t topk,
                       int32_t use_shared, float scale, int32_t num_items, int32_t *work_counter) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *s_tot = reinterpret_cast<float *>(sm + Smem::TOT);
    float *s_scale = reinterpret_cast<float *>(sm + Smem::SCALE);
    const uint32_t bar0 = smem_u32(sm + Smem::BAR);
    auto bar = [&](int i) { return bar0 + 8u * i; };
    uint32_t *s_slot = reinterpret_cast<uint32_t *>(sm + Smem::MISC);
    int *s_abort = reinterpret_cast<int *>(sm + Smem::MISC + 8);
    int *s_segq = reinterpret_cast<int *>(sm + Smem::SEGQ);

    const int tid = threadIdx.x, warp = tid >> 5;
    const __nv_bfloat16 *gg = static_cast<const __nv_bfloat16 *>(a.g);
    const int P = N + use_shared;

    auto meta_tok = [&](int stage) { return reinterpret_cast<int *>(sm + Smem::META + stage * Smem::META_STAGE); };
    auto meta_e = [&](int stage) {
        return reinterpret_cast<float *>(sm + Smem::META + stage * Smem::META_STAGE + 512);
    };
    auto meta_hdr = [&](int stage) {
        return reinterpret_cast<int *>(sm + Smem::META + stage * Smem::META_STAGE + 1024);
    };

    // ---- set-up ------------------------------------------------------------
    if (warp == 0) tmem_alloc(smem_u32(s_slot), kTmemCols);
    if (tid == 0) {
        mbar_init(bar(kBarT), kTrfThreads);
        mbar_init(bar(kBarSc0), KC);
        mbar_init(bar(kBarSc1), KC);
        mbar_init(bar(kBarS), 32 * kEpiWarps);
        mbar_init(bar(kBarA), 1);
        mbar_init(bar(kBarQK), 1);
        mbar_init(bar(kBarP), 32 * kEpiWarps);
        mbar_init(bar(kBarO), 1);
        mbar_init(bar(kBarOf0), 32 * kEpiWarps);
        mbar_init(bar(kBarOf1), 32 * kEpiWarps);
        mbar_init(bar(kBarV0), 1);
        mbar_init(bar(kBarV1), 1);
        mbar_init(bar(kBarVL0), 1);
        mbar_init(bar(kBarVL1), 1);
        for (int i = 0; i < kMetaStages; ++i) {
            mbar_init(bar(kBarMR + i), 32);
            mbar_init(bar(kBarMF + i), 32 * kEpiWarps);
        }
        for (int i = 0; i < kSegSlots; ++i) {
            mbar_init(bar(kBarSegF + i), 1);
            mbar_init(bar(kBarSegE + i), 32 * kEpiWarps + kTrfThreads);
        }
        mbar_fence_init();
        *s_abort = 0;
    }
    if (KC < 128) {  // Kt is also the M = 128 operand of the state pass: its second atom stays 0
        for (int x = tid; x < kC * 8; x += kThreads) {
            const int r = x / 8, chunk = x % 8;
            *reinterpret_cast<uint4 *>(sm + Smem::K + (r >> 3) * 2048 + 1024 + (r & 7) * 128 + chunk * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    fence_before();
    fence_proxy_async();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_slot;

    // The roles walk the same sequence of work items, each at its own pace: the
    // loader claims the items and posts them through the segment ring; every
    // per-chunk barrier counts chunks globally (g), so a role can be in the
    // next segment while another finishes the previous one.
    uint32_t gch = 0;  // chunks of earlier segments: barrier phase parity base
    bool failed = false;
    if (warp >= kEpiWarps + kTrfWarps) {
        // =================== loader warps ===================
        reg_dealloc<kRegsLdr>();
        const int lw = warp - kEpiWarps - kTrfWarps, lane = tid & 31;
        if (lw == 0) {
            // Work items -> segment ring; row metadata of every chunk -> meta
            // ring (lane l: rows 4l..4l+3), with an L2 prefetch of those rows of
            // q, k, g and v: the ring runs two to four chunks ahead of the
            // transform, so its row loads find them in L2 instead of waiting on
            // DRAM.  After the last item, one more stage whose header tells the
            // gather warps to stop.
            const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(a.v);
            uint32_t g = 0;
            for (int sidx = 0;; ++sidx) {
                int item = 0;
                if (lane == 0) {
                    item = *(volatile int *)s_abort ? num_items : atomicAdd(work_counter, 1);
                    if (item < num_items) item = queue_item(item, a.num_seqs * H, N, use_shared);
                }
                item = __shfl_sync(0xffffffffu, item, 0);
                const bool stop = item >= num_items;
                Segment seg{};
                int pad_base = 0;
                if (!stop) {
                    seg = decode_segment<MASKED>(a, item, H, N, use_shared);
                    pad_base = __ldcg(a.pad_off + item);
                }
                const int slot = sidx % kSegSlots;
                bool ok = sidx < kSegSlots ||
                          mbar_wait_bounded(bar(kBarSegE + slot), ((sidx / kSegSlots) - 1) & 1, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
                if (lane == 0) {
                    int *d = s_segq + slot * 8;
                    d[0] = stop ? -1 : item;
                    d[1] = seg.b;
                    d[2] = seg.h;
                    d[3] = seg.slot;
                    d[4] = seg.base;
                    d[5] = seg.len;
                    d[6] = pad_base;
                    d[7] = seg.shared ? 1 : 0;
                    mbar_arrive(bar(kBarSegF + slot));
                }
                const int nst = stop ? 1 : (seg.len + kC - 1) / kC;
                const __nv_bfloat16 *pq = static_cast<const __nv_bfloat16 *>(seg.shared && a.qs ? a.qs : a.q);
                const __nv_bfloat16 *pk = static_cast<const __nv_bfloat16 *>(seg.shared && a.ks ? a.ks : a.k);
                for (int n = 0; n < nst; ++n, ++g) {
                    const int st = g % kMetaStages;
                    ok = g < kMetaStages ||
                         mbar_wait_bounded(bar(kBarMF + st), ((g / kMetaStages) - 1) & 1, kWaitNs);
                    if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = 4 * lane + j;
                        const RowMeta m = stop ? RowMeta{-1, 0.f} : row_meta<MASKED>(a, seg, n * kC + r, H, topk);
                        meta_tok(st)[r] = m.t;
                        meta_e(st)[r] = m.e;
                        if (m.t >= 0) {
                            const int64_t th = (int64_t)m.t * H + seg.h;
                            prefetch_l2(pq + th * KC, KC * 2);
                            prefetch_l2(pk + th * KC, KC * 2);
                            prefetch_l2(gg + th * KC, KC * 2);
                            prefetch_l2(gv + th * DV, DV * 2);
                        }
                    }
                    if (lane == 0) {
                        int *hd = meta_hdr(st);
                        hd[0] = stop ? 1 : 0;
                        hd[1] = seg.h;
                        hd[2] = seg.shared ? 1 : 0;
                    }
                    mbar_arrive(bar(kBarMR + st));
                }
                if (failed || stop) break;
            }
        } else if (lw == 1) {
            // The V rows of every chunk into V0 / V1 once the chunk two back has
            // been consumed.  Lane l gathers rows 4l..4l+3 (rows past the
            // segment's end copy token row 0: their Kt rows are zero, so they add
            // nothing).
            int64_t last = -1;  // last chunk whose copies this warp issued
            const uint32_t off = (uint32_t)(lane >> 1) * 2048 + (uint32_t)(lane & 1) * 512;
            for (uint32_t g = 0;; ++g) {
                const int st = g % kMetaStages;
                bool ok = mbar_wait_bounded(bar(kBarMR + st), (g / kMetaStages) & 1, kWaitNs);
                if (ok && g >= 2)
                    ok = mbar_wait_bounded(bar((g & 1) ? kBarV1 : kBarV0), ((g - 2) >> 1) & 1, kWaitNs);
                // Queue behind the output store of chunk g - 3 (the TMA engine works
                // in order: the epilogue's next state-row pass waits for that store
                // to have read its staging tile, not for these gathers).
                if (ok && g >= 3)
                    ok = mbar_wait_bounded(bar(kBarMF + (g - 3) % kMetaStages), ((g - 3) / kMetaStages) & 1, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
                const int *hd = meta_hdr(st);
                if (hd[0]) break;
                const int h = hd[1];
                const int *tok = meta_tok(st);
                int rr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = tok[4 * lane + j];
                    rr[j] = t >= 0 ? t * H + h : 0;
                }
                const uint32_t mb = bar((g & 1) ? kBarVL1 : kBarVL0);
                if (lane == 0) mbar_arrive_expect_tx(mb, kC * DV * 2);
                __syncwarp();
                const uint32_t dst = smem_u32(sm + ((g & 1) ? Smem::V1 : Smem::V0)) + off;
#pragma unroll
                for (int at = 0; at < DV / 64; ++at)
                    tma_gather4(&maps.v, dst + at * 1024, mb, at * 64, rr[0], rr[1], rr[2], rr[3]);
                last = g;
            }
            // no copy of this warp may still be writing shared memory when the CTA exits
            if (last >= 0 &&
                !mbar_wait_bounded(bar((last & 1) ? kBarVL1 : kBarVL0), (uint32_t)((last >> 1) & 1), kWaitNs))
                failed = true;
        } else if (lw == 2) {
            // The tensor-core products of every chunk, issued by lane 0 as their
            // operands become ready: A = Qt Kt^T once Qt, Kt are written (P of
            // the previous chunk was read out of A before its P V was issued);
            // S += Kt^T V once the state rows are rescaled and V has landed;
            // O = Qt S' once that O buffer has been read out for chunk g - 2;
            // O += P V once P is written.
            const uint32_t q0 = smem_u32(sm + Smem::Q), k0 = smem_u32(sm + Smem::K);
            const uint32_t p0 = smem_u32(sm + Smem::P), s0 = smem_u32(sm + Smem::S);
            constexpr uint32_t idA = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idS = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t idO = idesc_bf16(128, DV, 0, 1);
            for (uint32_t g = 0;; ++g) {
                const int st = g % kMetaStages;
                bool ok = mbar_wait_bounded(bar(kBarMR + st), (g / kMetaStages) & 1, kWaitNs);
                if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
                if (meta_hdr(st)[0]) break;
                const uint32_t v0 = smem_u32(sm + ((g & 1) ? Smem::V1 : Smem::V0));
                const uint32_t tO = tmem + ((g & 1) ? kTmemO1 : kTmemO0);
                ok = mbar_wait_bounded(bar(kBarT), g & 1, kWaitNs);
                if (ok && lane == 0) {
                    fence_after();
#pragma unroll 1
                    for (int k16 = 0; k16 < KC; k16 += 16) {
                        const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                        mma_bf16(tmem + kTmemA, desc_sw128(q0 + ko, 16, 2048), desc_sw128(k0 + ko, 16, 2048), idA,
                                 k16 > 0);
                    }
                    commit(bar(kBarA));
                }
                __syncwarp();
                ok = ok && mbar_wait_bounded(bar(kBarS), g & 1, kWaitNs) &&
                     mbar_wait_bounded(bar((g & 1) ? kBarVL1 : kBarVL0), (g >> 1) & 1, kWaitNs);
                if (ok && lane == 0) {
                    fence_after();
#pragma unroll 1
                    for (int k16 = 0; k16 < kC; k16 += 16) {
                        const uint32_t ro = (k16 / 8) * 2048;
                        mma_bf16(tmem + kTmemS, desc_sw128(k0 + ro, 1024, 2048), desc_sw128(v0 + ro, 1024, 2048), idS,
                                 1);
                    }
                }
                __syncwarp();
                // two read-out barriers by chunk parity: at a segment's end the
                // epilogue reads out the last O without waiting for this warp
                if (ok && g >= 2) ok = mbar_wait_bounded(bar((g & 1) ? kBarOf1 : kBarOf0), ((g - 2) >> 1) & 1, kWaitNs);
                if (ok && lane == 0) {
                    fence_after();
#pragma unroll 1
                    for (int k16 = 0; k16 < KC; k16 += 16) {
                        const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                        mma_bf16(tO, desc_sw128(q0 + ko, 16, 2048), desc_sw128(s0 + (k16 / 8) * 2048, 1024, 2048), idO,
                                 k16 > 0);
                    }
                    commit(bar(kBarQK));
                }
                __syncwarp();
                ok = ok && mbar_wait_bounded(bar(kBarP), g & 1, kWaitNs);
                if (ok && lane == 0) {
                    fence_after();
#pragma unroll 1
                    for (int k16 = 0; k16 < kC; k16 += 16) {
                        const uint32_t ko = (k16 / 64) * 1024 + (k16 % 64) * 2;
                        mma_bf16(tO, desc_sw128(p0 + ko, 16, 2048), desc_sw128(v0 + (k16 / 8) * 2048, 1024, 2048), idO,
                                 1);
                    }
                    commit(bar(kBarO));
                    commit(bar((g & 1) ? kBarV1 : kBarV0));
                }
                if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
            }
        }
    } else if (warp >= kEpiWarps) {
        // =================== transform warps ===================
        reg_alloc<kRegsTrf>();
        const int tt = tid - 32 * kEpiWarps;  // 0..255
        constexpr int CG = KC / 8, NRB = kTrfThreads / CG, RPT = kC / NRB;
        const int cg = tt % CG, rb = tt / CG, col0 = cg * 8;
        for (int sidx = 0;; ++sidx) {
            const int slot = sidx % kSegSlots;
            const bool ok = mbar_wait_bounded(bar(kBarSegF + slot), (sidx / kSegSlots) & 1, kWaitNs);
            if (named_sync_or(1, kTrfThreads, !ok)) { failed = true; break; }
            const int *d = s_segq + slot * 8;
            const int item = d[0], seg_h = d[2], seg_len = d[5];
            const bool seg_shared = d[7] != 0;
            mbar_arrive(bar(kBarSegE + slot));
            if (item < 0) break;
            const int nch = (seg_len + kC - 1) / kC;
            const __nv_bfloat16 *qsrc = static_cast<const __nv_bfloat16 *>(seg_shared && a.qs ? a.qs : a.q);
            const __nv_bfloat16 *ksrc = static_cast<const __nv_bfloat16 *>(seg_shared && a.ks ? a.ks : a.k);
            uint4 rq[RPT], rk[RPT], rg[RPT];
            // raw g rows of chunk n (its metadata stage must have been written)
            auto load_g = [&](int n, uint4 (&dst)[RPT]) -> bool {
                const uint32_t g = gch + n;
                const bool ok = mbar_wait_bounded(bar(kBarMR + g % kMetaStages), (g / kMetaStages) & 1, kWaitNs);
                const int *tok = meta_tok(g % kMetaStages);
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const int t = ok ? tok[rb * RPT + i] : -1;
                    dst[i] = t >= 0 ? ldg_stream(gg + ((int64_t)t * H + seg_h) * KC + col0)
                                    : make_uint4(0, 0, 0, 0);
                }
                return ok;
            };
            bool bad = false, seg_redo = false;
            if (nch > 0) bad = !load_g(0, rg);
            for (int n = 0; n < nch; ++n) {
                const uint32_t g_n = gch + n;
                const int mst = g_n % kMetaStages;
                const int *tok_n = meta_tok(mst);
                // pass 1: per-thread running sums of g over its rows -> block totals
                // (masking schedule: the rows of tokens that did not select this
                // partition get gate 0, i.e. no decay)
                {
                    if (MASKED) {
                        const float *me = meta_e(mst);
#pragma unroll
                        for (int i = 0; i < RPT; ++i)
                            if (me[rb * RPT + i] < 0.f) rg[i] = make_uint4(0, 0, 0, 0);
                    }
                    F2 run[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                    for (int i = 0; i < RPT; ++i) {
                        // this row's raw q, k (used by pass 2), issued between the sums
                        const int t = tok_n[rb * RPT + i];
                        if (t >= 0) {
                            const int64_t ro = ((int64_t)t * H + seg_h) * KC + col0;
                            rq[i] = ldg_stream(qsrc + ro);
                            rk[i] = ldg_stream(ksrc + ro);
                        } else {
                            rq[i] = rk[i] = make_uint4(0, 0, 0, 0);
                        }
                        const uint32_t w[4] = {rg[i].x, rg[i].y, rg[i].z, rg[i].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float lo, hi;
                            unpack2(w[j], lo, hi);
                            run[j] = add2(run[j], f2(lo, hi));
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 x = f2_get(run[j]);
                        s_tot[rb * 128 + col0 + 2 * j] = x.x;
                        s_tot[rb * 128 + col0 + 2 * j + 1] = x.y;
                    }
                }
                if (named_sync_or(1, kTrfThreads, bad)) { failed = true; break; }
                // the next chunk's metadata, for its g rows loaded inside pass 2
                const int *tok_next = nullptr;
                if (n + 1 < nch) {
                    const uint32_t g1 = g_n + 1;
                    bad = !mbar_wait_bounded(bar(kBarMR + g1 % kMetaStages), (g1 / kMetaStages) & 1, kWaitNs);
                    if (!bad) tok_next = meta_tok(g1 % kMetaStages);
                }
                float *s_fmid = s_scale + (g_n & 1) * 256, *s_beta = s_fmid + 128;
                bool out_of_range = false;
                if (tt < KC) {  // per-column exclusive scan over row blocks
                    float acc = 0.f, gmid = 0.f;
                    for (int r2 = 0; r2 < NRB; ++r2) {
                        const float x = s_tot[r2 * 128 + tt];
                        s_tot[r2 * 128 + tt] = acc;
                        acc += x;
                        if ((r2 + 1) * RPT - 1 == kMid) gmid = acc;
                    }
                    s_fmid[tt] = expf(gmid);
                    s_beta[tt] = expf(acc - gmid);
                    s_tot[32 * 128 + tt] = gmid * kLog2e;
                    // |G_r - G_m| over the chunk: with log-gates <= 0 (decays in
                    // (0, 1]) G_r falls monotonically from 0, so it is at most
                    // max(|G_m|, |G_last - G_m|)
                    out_of_range = fmaxf(fabsf(gmid), fabsf(acc - gmid)) > kGateRange;
                    // the state rows can be rescaled now (two barriers by chunk parity:
                    // this role may reach the next chunk's scan before the epilogue
                    // has waited for this one)
                    mbar_arrive(bar((g_n & 1) ? kBarSc1 : kBarSc0));
                }
                // A chunk past the gate range: the segment is finished as usual
                // (its results are overwritten) and queued once for the exact
                // per-token recomputation.
                if (named_sync_or(1, kTrfThreads, out_of_range) && !seg_redo) {
                    seg_redo = true;
                    if (tt == 0) {
                        atomicOr(a.flags, SSE_DEVICE_RECOMPUTED);
                        a.redo_list[atomicAdd(a.flags + 1, 1)] = item;
                    }
                }
                // Qt / Kt tiles are free once the products of chunk g_n - 1 read them
                if (g_n >= 1) bad |= !mbar_wait_bounded(bar(kBarQK), (g_n - 1) & 1, kWaitNs);
                // pass 2: Qt, Kt rows (bf16) into their tiles.  The read weight
                // e * scale is applied to the output rows by the epilogue.  The decay
                // factors are rounded to bf16 and multiplied into the bf16 q / k pairs
                // with packed bf16 products.
                {
                    // run = (G_r - G_m) log2(e), advanced row by row
                    F2 run[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        run[j] = f2(fmaf(s_tot[rb * 128 + col0 + 2 * j], kLog2e, -s_tot[32 * 128 + col0 + 2 * j]),
                                    fmaf(s_tot[rb * 128 + col0 + 2 * j + 1], kLog2e,
                                         -s_tot[32 * 128 + col0 + 2 * j + 1]));
                    const F2 l2e = f2(kLog2e, kLog2e);
                    const float *me = meta_e(mst);
#pragma unroll
                    for (int i = 0; i < RPT; ++i) {
                        const int r = rb * RPT + i;
                        const float e = MASKED ? fmaxf(me[r], 0.f) : me[r];
                        const F2 e2 = f2(e, e);
                        const uint32_t wg4[4] = {rg[i].x, rg[i].y, rg[i].z, rg[i].w};
                        const uint32_t wq4[4] = {rq[i].x, rq[i].y, rq[i].z, rq[i].w};
                        const uint32_t wk4[4] = {rk[i].x, rk[i].y, rk[i].z, rk[i].w};
                        uint32_t pq[4], pk[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float g0, g1;
                            unpack2(wg4[j], g0, g1);
                            run[j] = fma2(f2(g0, g1), l2e, run[j]);
                            const float2 dd = f2_get(run[j]);
                            pq[j] = bf16x2_mul(wq4[j], pack_bf16x2(ex2(dd.x), ex2(dd.y)));
                            const float2 kf = f2_get(mul2(e2, f2(ex2(-dd.x), ex2(-dd.y))));
                            pk[j] = bf16x2_mul(wk4[j], pack_bf16x2(kf.x, kf.y));
                        }
                        // row i of the next chunk's g, into the registers just consumed
                        {
                            const int t1 = tok_next ? tok_next[r] : -1;
                            rg[i] = t1 >= 0 ? ldg_stream(gg + ((int64_t)t1 * H + seg_h) * KC + col0)
                                            : make_uint4(0, 0, 0, 0);
                        }
                        *reinterpret_cast<uint4 *>(sm + Smem::Q + tile_off(r, col0)) =
                            make_uint4(pq[0], pq[1], pq[2], pq[3]);
                        *reinterpret_cast<uint4 *>(sm + Smem::K + tile_off(r, col0)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                fence_proxy_async();
                if (named_sync_or(1, kTrfThreads, bad)) { failed = true; break; }
#ifdef SSE_FAULT_INJECT
                if (!(g_fault_mode == 1 && blockIdx.x == 0 && g_n == 0))
#endif
                mbar_arrive(bar(kBarT));
            }
            if (failed) break;
            gch += nch;
        }
    } else {
        reg_dealloc<kRegsEpi>();
        for (int sidx = 0;; ++sidx) {
            const int slot = sidx % kSegSlots;
            const bool ok = mbar_wait_bounded(bar(kBarSegF + slot), (sidx / kSegSlots) & 1, kWaitNs);
            if (named_sync_or(2, 32 * kEpiWarps, !ok)) { failed = true; break; }
            const int *d = s_segq + slot * 8;
            const int item = d[0];
            Segment seg;
            seg.b = d[1];
            seg.h = d[2];
            seg.slot = d[3];
            seg.base = d[4];
            seg.len = d[5];
            const int pad_base = d[6];
            seg.shared = d[7] != 0;
            mbar_arrive(bar(kBarSegE + slot));
            if (item < 0) break;
            const int nch = (seg.len + kC - 1) / kC;
            const int64_t state_off = (((int64_t)seg.b * H + seg.h) * P + seg.slot) * (int64_t)KC * DV;
            // =================== epilogue warps ===================
            const int row = tid;  // TMEM lane
            const uint32_t lb = (uint32_t)(32 * warp) << 16;
            const uint32_t tA = tmem + lb + kTmemA, tS = tmem + lb + kTmemS;
            // initial state -> TMEM
            if (row < KC) {
#pragma unroll 1  // once per segment: rolled, small code
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    uint32_t r[32];
                    const float *src = a.init ? a.init + state_off + (int64_t)row * DV + c0 : nullptr;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float4 f = src ? *reinterpret_cast<const float4 *>(src + i) : make_float4(0, 0, 0, 0);
                        r[i] = __float_as_uint(f.x);
                        r[i + 1] = __float_as_uint(f.y);
                        r[i + 2] = __float_as_uint(f.z);
                        r[i + 3] = __float_as_uint(f.w);
                    }
                    tmem_st32(tS + c0, r);
                }
                tmem_wait_st();
            }
            float p_pending = 1.f;
            // Output of chunk n_o (O buffer of its parity), written one chunk late so
            // that it overlaps the transform's compute: each thread scales its TMEM
            // row of O by the read weight e * scale and stores it as bf16 into the
            // S' tile (free once the O = Qt S' product of the following chunk has
            // completed), laid out as the tensor map's 64-column boxes with the
            // 128-byte swizzle (conflict-free 16-byte stores).  One thread then
            // hands the whole chunk to the TMA engine: the work item's rows of the
            // partial buffer are contiguous and padded to whole chunks, so the chunk
            // is DV/64 box stores.  The staging tile is reused only after
            // bulk_wait_read().
            auto write_out = [&](int n_o, bool pend) -> bool {
                const int st = (gch + n_o) % kMetaStages;
                const float w = (MASKED ? fmaxf(meta_e(st)[row], 0.f) : meta_e(st)[row]) * scale;
                const F2 w2 = f2(w, w);
                const uint32_t tO = tmem + lb + (((gch + n_o) & 1) ? kTmemO1 : kTmemO0);
                unsigned char *stg = sm + Smem::S;
#pragma unroll 1  // one 32-column block per iteration: keeps the hot code small
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tO + c0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int col = c0 + 8 * i;
                        const int ch = (col % 64) / 8;
                        uint32_t o4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 x = f2_get(mul2(w2, f2_bits(r[8 * i + 2 * u], r[8 * i + 2 * u + 1])));
                            o4[u] = pack_bf16x2(x.x, x.y);
                        }
                        *reinterpret_cast<uint4 *>(stg + (col / 64) * (kC * 128) + row * 128 + ((ch ^ (row & 7)) << 4)) =
                            make_uint4(o4[0], o4[1], o4[2], o4[3]);
                    }
                }
                fence_before();
                mbar_arrive(bar(((gch + n_o) & 1) ? kBarOf1 : kBarOf0));  // O may be overwritten now
                fence_proxy_async();
                if (named_sync_or(3, 32 * kEpiWarps, pend)) return true;
                if (tid == 0) {
#pragma unroll
                    for (int atom = 0; atom < DV / 64; ++atom)
                        tma_store_2d(&part_map, smem_u32(stg + atom * (kC * 128)), atom * 64, pad_base + n_o * kC);
                    bulk_commit();
                }
                // the chunk's metadata stage is free again, and its output store is
                // queued on the TMA engine (the V gathers of chunk n_o + 3 wait for this)
                mbar_arrive(bar(kBarMF + st));
                return false;
            };
            // A wait that runs out of time sets `pend` in the threads that saw it;
            // the epilogue warps take every decision to stop together, at one of
            // their named barriers (bar.red.or), so none is left waiting there.
            bool pend = false;
            for (int n = 0; n < nch; ++n) {
                const uint32_t g_n = gch + n;
                // the state-row pass needs only the chunk's gate scan; it overlaps
                // the transform's Qt / Kt pass
                pend |= !mbar_wait_bounded(bar((g_n & 1) ? kBarSc1 : kBarSc0), (g_n >> 1) & 1, kWaitNs);
                if (n >= 1) {
                    pend |= !mbar_wait_bounded(bar(kBarO), (g_n - 1) & 1, kWaitNs);
                    fence_after();
                }
                // state rows: S_stored *= exp(G_m) * p; bf16 copy -> S' tile, once the
                // TMA engine has read the previous chunk's staged output from it
                bulk_wait_read();
                if (named_sync_or(2, 32 * kEpiWarps, pend)) { failed = true; break; }
                const float *s_fmid = s_scale + (g_n & 1) * 256, *s_beta = s_fmid + 128;
                if (row < KC) {
                    // S_stored * p is the state itself, then * exp(G_m): the two
                    // factors are applied one after the other because their product
                    // (down to e^-160 within the gate range) would underflow
                    const float fm = s_fmid[row];
                    const F2 pp2 = f2(p_pending, p_pending), fm2 = f2(fm, fm);
#pragma unroll 1  // one 32-column block per iteration: keeps the hot code small
                    for (int c0 = 0; c0 < DV; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(tS + c0, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 x = f2_get(mul2(mul2(f2_bits(r[i], r[i + 1]), pp2), fm2));
                            r[i] = __float_as_uint(x.x);
                            r[i + 1] = __float_as_uint(x.y);
                        }
                        tmem_st32(tS + c0, r);
#pragma unroll
                        for (int i = 0; i < 32; i += 8)
                            *reinterpret_cast<uint4 *>(sm + Smem::S + tile_off(row, c0 + i)) = make_uint4(
                                pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                                pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                    }
                    tmem_wait_st();
                    p_pending = s_beta[row];
                }
                fence_proxy_async();
                fence_before();
                mbar_arrive(bar(kBarS));
                // P = causal mask of A, bf16
                pend |= !mbar_wait_bounded(bar(kBarA), g_n & 1, kWaitNs);
                fence_after();
                // warp w holds rows 32w..32w+31: column blocks left of the diagonal
                // block are copied, the diagonal block is masked, the rest is 0
#pragma unroll 1  // one 32-column block per iteration: keeps the hot code small
                for (int c0 = 0; c0 < kC; c0 += 32) {
                    if (c0 > 32 * warp) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8)
                            *reinterpret_cast<uint4 *>(sm + Smem::P + tile_off(row, c0 + i)) = make_uint4(0, 0, 0, 0);
                        continue;
                    }
                    uint32_t r[32];
                    tmem_ld32(tA + c0, r);
                    tmem_wait_ld();
                    const bool diag = c0 == 32 * warp;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        float f[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            f[j] = (!diag || c0 + i + j <= row) ? __uint_as_float(r[i + j]) : 0.f;
                        *reinterpret_cast<uint4 *>(sm + Smem::P + tile_off(row, c0 + i)) =
                            make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                       pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
                fence_proxy_async();
                fence_before();
                mbar_arrive(bar(kBarP));
                if (n >= 1) {  // output of the previous chunk, staged in S' once O = Qt S' of this one is done
                    pend |= !mbar_wait_bounded(bar(kBarQK), g_n & 1, kWaitNs);
                    fence_after();
                    if (write_out(n - 1, pend)) { failed = true; break; }
                    pend = false;
                }
            }
            if (!failed && nch > 0) {
                const uint32_t g_l = gch + nch - 1;
                pend |= !mbar_wait_bounded(bar(kBarO), g_l & 1, kWaitNs);
                fence_after();
                // the staging tile is free once the previous chunk's store has read it
                bulk_wait_read();
                if (named_sync_or(2, 32 * kEpiWarps, pend) || write_out(nch - 1, false)) failed = true;
            }
            bulk_wait_all();
            // final state = p * S_stored
            if (!failed && a.final_state && row < KC) {
#pragma unroll 1  // once per segment: rolled, small code
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tS + c0, r);
                    tmem_wait_ld();
                    float4 *o4 = reinterpret_cast<float4 *>(a.final_state + state_off + (int64_t)row * DV + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        o4[i] = make_float4(__uint_as_float(r[4 * i]) * p_pending,
                                            __uint_as_float(r[4 * i + 1]) * p_pending,
                                            __uint_as_float(r[4 * i + 2]) * p_pending,
                                            __uint_as_float(r[4 * i + 3]) * p_pending);
                }
            }
            fence_before();
                if (failed) break;
            gch += nch;
        }
    }
    if (failed) {
        atomicOr(a.flags, SSE_DEVICE_TIMEOUT);
        *s_abort = 1;
    }
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Exact per-token recomputation of the work items the tensor-core kernel put
// on the redo list (a chunk whose summed log-gate left the factorised form's
// range, kGateRange).  The recurrence of eqs. 13-14 is evaluated one row at a
// time in float32 -- decay of the state rows, write of e k^T v, read of
// w q S -- with exp(g) taken per row, so any decay in (0, 1] is exact to
// float32 rounding.  Each item's partial rows (pad_off[item] + row) and its
// final state overwrite what the tensor-core kernel wrote.  CTAs stride over
// the list; an empty list costs one launch that reads one word.
// Thread layout: DV/4 column quads x R row groups, KC/R state rows each.
template <int KC, int DV, bool MASKED>
__global__ void __launch_bounds__(256)
segment_redo_kernel(ForwardArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared, float scale) {
    constexpr int D4 = DV / 4, R = 256 / D4, RPT = KC / R, kBatch = 32;
    __shared__ float s_q[KC], s_k[KC], s_a[KC], s_v[DV];
    __shared__ float s_red[R][DV];
    __shared__ int s_tok[kBatch];
    __shared__ float s_e[kBatch];
    const int tid = threadIdx.x, cq = tid % D4, rg = tid / D4, col = 4 * cq;
    const int count = *(volatile const int32_t *)(a.flags + 1);
    const int P = N + use_shared;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *kk = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
    const __nv_bfloat16 *g = static_cast<const __nv_bfloat16 *>(a.g);
    __nv_bfloat16 *part = static_cast<__nv_bfloat16 *>(a.part_routed);
    for (int li = blockIdx.x; li < count; li += gridDim.x) {
        const int item = __ldcg(a.redo_list + li);
        const Segment seg = decode_segment<MASKED>(a, item, H, N, use_shared);
        const int64_t state_off = (((int64_t)seg.b * H + seg.h) * P + seg.slot) * (int64_t)KC * DV;
        const int64_t row0 = __ldcg(a.pad_off + item);
        const __nv_bfloat16 *qsrc = seg.shared && a.qs ? static_cast<const __nv_bfloat16 *>(a.qs) : q;
        const __nv_bfloat16 *ksrc = seg.shared && a.ks ? static_cast<const __nv_bfloat16 *>(a.ks) : kk;
        float4 st[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int r = rg + m * R;
            st[m] = a.init ? *reinterpret_cast<const float4 *>(a.init + state_off + (int64_t)r * DV + col)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int i0 = 0; i0 < seg.len; i0 += kBatch) {
            __syncthreads();  // the previous batch's metadata has been read
            if (tid < kBatch) {
                const RowMeta mt = row_meta<MASKED>(a, seg, i0 + tid, H, topk);
                s_tok[tid] = mt.t;
                s_e[tid] = mt.e;
            }
            __syncthreads();
            const int nb = min(kBatch, seg.len - i0);
            for (int j = 0; j < nb; ++j) {
                const int t = s_tok[j];
                const float e = s_e[j];
                if (MASKED && e < 0.f) continue;  // not selected: no decay, no write, no read
                const int64_t th = (int64_t)t * H + seg.h;
                for (int r = tid; r < KC; r += 256) {
                    s_q[r] = e * scale * __bfloat162float(qsrc[th * KC + r]);
                    s_k[r] = e * __bfloat162float(ksrc[th * KC + r]);
                    s_a[r] = expf(__bfloat162float(g[th * KC + r]));
                }
                for (int c2 = tid; c2 < DV; c2 += 256) s_v[c2] = __bfloat162float(v[th * DV + c2]);
                __syncthreads();
                const float4 v4 = *reinterpret_cast<const float4 *>(s_v + col);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int m = 0; m < RPT; ++m) {
                    const int r = rg + m * R;
                    const float ar = s_a[r], kr = s_k[r], qr = s_q[r];
                    st[m].x = fmaf(ar, st[m].x, kr * v4.x);
                    st[m].y = fmaf(ar, st[m].y, kr * v4.y);
                    st[m].z = fmaf(ar, st[m].z, kr * v4.z);
                    st[m].w = fmaf(ar, st[m].w, kr * v4.w);
                    acc.x = fmaf(qr, st[m].x, acc.x);
                    acc.y = fmaf(qr, st[m].y, acc.y);
                    acc.z = fmaf(qr, st[m].z, acc.z);
                    acc.w = fmaf(qr, st[m].w, acc.w);
                }
                *reinterpret_cast<float4 *>(&s_red[rg][col]) = acc;
                __syncthreads();
                for (int c2 = tid; c2 < DV; c2 += 256) {
                    float o = 0.f;
#pragma unroll
                    for (int r2 = 0; r2 < R; ++r2) o += s_red[r2][c2];
                    part[(row0 + i0 + j) * DV + c2] = __float2bfloat16_rn(o);
                }
                __syncthreads();  // s_q .. s_red are rewritten by the next row
            }
        }
        if (a.final_state) {
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                const int r = rg + m * R;
                *reinterpret_cast<float4 *>(a.final_state + state_off + (int64_t)r * DV + col) = st[m];
            }
        }
    }
}

// out[row, :] = sum over the row's NC bf16 partial rows rec_pos[row * NC + j]
// (routed contributions j < k, then the shared one), 8 columns per thread,
// fp32 accumulation in a fixed order.  NC is a template constant so that a
// thread issues all NC position loads, then all NC row loads, before it sums
// (measured: 99 -> 87 us on the 8 x 4096-token layer, 92 % of the HBM copy
// rate; taking two or four pieces per thread was no faster, or slower).
template <int NC>
__global__ void __launch_bounds__(256)
gather_combine_kernel(const __nv_bfloat16 *part, const int32_t *rec_pos, int64_t rows,
                      int32_t d, __nv_bfloat16 *__restrict__ out) {
    const int cpr = d / 8;
    const int64_t total = rows * cpr;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = x / cpr;
        const int ch = (int)(x - row * cpr);
        int32_t pr[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) pr[j] = __ldcg(rec_pos + row * NC + j);
        uint4 pv[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j)
            pv[j] = __ldcg(reinterpret_cast<const uint4 *>(part + (int64_t)pr[j] * d + ch * 8));
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const uint32_t wv[4] = {pv[j].x, pv[j].y, pv[j].z, pv[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo, hi;
                unpack2(wv[i], lo, hi);
                acc[2 * i] += lo;
                acc[2 * i + 1] += hi;
            }
        }
        *reinterpret_cast<uint4 *>(out + row * d + ch * 8) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null when unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

template <int KC, int DV, bool MASKED>
cudaError_t launch_t(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    static bool attr_set = false;  // benign race: every caller sets the same value
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunked_forward_kernel<KC, DV, MASKED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t nseg = (int64_t)a.num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    if (nseg == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // the work counter (a.flags[2]) and the redo list's length (a.flags[1])
    // start at zero with the flags words, cleared by the caller before routing
    int32_t *counter = a.flags + 2;

    // The partial buffer as a 2-D tensor [part_rows, DV] of bf16, stored in
    // boxes of 64 columns x one chunk of rows with the 128-byte swizzle.
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    // v as [T * H, d] bf16, gathered in boxes of 64 columns x 1 row with the
    // 128-byte swizzle (no rows: never read, left zero).
    const int64_t th_rows = a.total_tokens * cfg.num_heads;
    auto row_map = [&](CUtensorMap *m, const void *base, int width) -> bool {
        memset(m, 0, sizeof *m);
        if (th_rows == 0) return true;
        cuuint64_t d[2] = {(cuuint64_t)width, (cuuint64_t)th_rows};
        cuuint64_t st[1] = {(cuuint64_t)width * 2};
        cuuint32_t bx[2] = {64, 1};
        cuuint32_t es[2] = {1, 1};
        return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), d, st, bx, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    RowMaps maps;
    if (!row_map(&maps.v, a.v, DV)) return cudaErrorInvalidValue;
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)DV, (cuuint64_t)a.part_rows};
    cuuint64_t strides[1] = {(cuuint64_t)DV * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kC};
    cuuint32_t elem_strides[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.part_routed, dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    const int grid = (int)std::min<int64_t>(nseg, sms > 0 ? sms : 148);
    chunked_forward_kernel<KC, DV, MASKED><<<grid, kThreads, kSmemBytes, stream>>>(
        a, map, maps, cfg.num_heads, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale, (int32_t)nseg, counter);
    const int redo_grid = (int)std::min<int64_t>(nseg, 2 * (sms > 0 ? sms : 148));
    segment_redo_kernel<KC, DV, MASKED><<<redo_grid, 256, 0, stream>>>(a, cfg.num_heads, cfg.num_partitions,
                                                                       cfg.top_k, cfg.use_shared, cfg.scale);
    return cudaGetLastError();
}

}  // namespace

bool chunked_supported(const sse_config_t &cfg) {
    const bool c_ok = cfg.key_dim == 64 || cfg.key_dim == 128;
    const bool d_ok = cfg.value_dim == 64 || cfg.value_dim == 128;
    return cfg.dtype == SSE_BF16 && c_ok && d_ok;
}

// 256 bytes reserved (the work counter lives in the flags words), then the redo
// list (one entry per work item)
size_t chunked_extra_workspace(const sse_config_t &cfg, int64_t, int32_t num_seqs) {
    const int64_t nitems = (int64_t)num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    return 256 + (size_t)nitems * sizeof(int32_t);
}

cudaError_t launch_forward_chunked(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream,
                                   int *launches) {
    cudaError_t e;
    const bool m = cfg.algo == SSE_ALGO_MASKED;
    if (cfg.key_dim == 128 && cfg.value_dim == 128)
        e = m ? launch_t<128, 128, true>(cfg, a, stream) : launch_t<128, 128, false>(cfg, a, stream);
    else if (cfg.key_dim == 128 && cfg.value_dim == 64)
        e = m ? launch_t<128, 64, true>(cfg, a, stream) : launch_t<128, 64, false>(cfg, a, stream);
    else if (cfg.key_dim == 64 && cfg.value_dim == 128)
        e = m ? launch_t<64, 128, true>(cfg, a, stream) : launch_t<64, 128, false>(cfg, a, stream);
    else if (cfg.key_dim == 64 && cfg.value_dim == 64)
        e = m ? launch_t<64, 64, true>(cfg, a, stream) : launch_t<64, 64, false>(cfg, a, stream);
    else return cudaErrorInvalidValue;
    *launches += 2;  // the tensor-core kernel and the (usually empty) redo pass
    return e;
}

int64_t chunked_part_rows(const sse_config_t &cfg, int64_t total_tokens, int32_t num_seqs) {
    const int64_t nitems = (int64_t)num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    // masking schedule: every item is a whole sequence
    const int64_t per_token = cfg.algo == SSE_ALGO_MASKED ? cfg.num_partitions + cfg.use_shared
                                                          : cfg.top_k + cfg.use_shared;
    return total_tokens * cfg.num_heads * per_token + nitems * (kChunkRows - 1);
}

cudaError_t launch_gather_combine(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    const int ncon = cfg.top_k + cfg.use_shared;
    const int64_t rows = a.total_tokens * cfg.num_heads;
    if (rows == 0) return cudaSuccess;
    const int64_t work = rows * (cfg.value_dim / 8);
    const unsigned blocks = (unsigned)std::min<int64_t>((work + 255) / 256, 152 * 16);
    const __nv_bfloat16 *part = static_cast<const __nv_bfloat16 *>(a.part_routed);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
    const int32_t *rp = a.rec_pos;
    switch (ncon) {
#define SSE_COMBINE(NC) \
    case NC: gather_combine_kernel<NC><<<blocks, 256, 0, stream>>>(part, rp, rows, cfg.value_dim, out); break
        SSE_COMBINE(1); SSE_COMBINE(2); SSE_COMBINE(3); SSE_COMBINE(4); SSE_COMBINE(5);
        SSE_COMBINE(6); SSE_COMBINE(7); SSE_COMBINE(8); SSE_COMBINE(9);
#undef SSE_COMBINE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sse

#ifdef SSE_FAULT_INJECT
// Checked build only: sets the fault mode read by chunked_forward_kernel (0 =
// none, 1 = CTA 0 withholds its first transform arrival).  Returns the CUDA
// error of the copy.
extern "C" int sse_debug_set_fault(int mode) {
    return (int)cudaMemcpyToSymbol(sse::g_fault_mode, &mode, sizeof(int));
}
#endif
