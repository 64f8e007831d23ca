// delta.cu -- SSE on a gated delta-rule transition (CUDA cores, float32).
//
// The close-reading notes of "Scaling Linear Attention with Sparse State
// Expansion" name Gated DeltaNet's structured transition (section 2.1, eq. 6)
// as the alternative to GLA's diagonal decay and the combination as future
// work (section 6); DeltaNet's update is on the "动态线性注意力" page (section
// 2.1, eq. 4).  With the SSE router (eqs. 9-10), per token t and head h:
//
//   for i in T_t:  S_i <- alpha_t (I - e_t[i] beta_t k_t^T k_t) S_i + e_t[i] beta_t k_t^T v_t
//   shared:        S_N <- alpha_t (I - beta_t ks_t^T ks_t) S_N + beta_t ks_t^T v_t
//   o_t = sum_{i in T_t} e_t[i] (scale q_t) S_i + (scale qs_t) S_N
//
// alpha_t = exp(log_alpha_t) and beta_t are one scalar each per (token, head).
// Row by row: with w = k S (the state's answer to the key, before the step),
//   S[r, :] <- alpha S[r, :] + e beta k[r] (v - alpha w).
//
// Forward: one CTA per (sequence, head, partition) segment of the grouping
// (section 2.6, varlen schedule) and per shared (sequence, head), walking its
// rows in time order with the c x d state in registers (delta_cols_kernel for
// c = 128 and d in {64, 128}, delta_segment_kernel for the other shapes);
// read-outs go to the float32 partial slots that launch_combine sums (the
// recurrent path's).
// Decode: one CTA per (sequence, head) routes the token (warp-level softmax
// and top-k) and updates only the k + 1 selected states in place.
#include <algorithm>

#include "f32x2.cuh"
#include "sse_internal.cuh"

namespace sse {
namespace {

constexpr int kDThreads = 256;
constexpr int kDMaxRows = 16;  // state rows per thread

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Thread layout (both kernels): D4 = d/4 column quads x R = 256/D4 row groups;
// thread (rg, cq) holds rows rg, rg + R, ... (at most kDMaxRows) x 4 columns.
// Shared memory: s_k, s_q [c], s_v [d], s_w [d], s_cols [R][d].
template <int D4>
struct DeltaRow {
    static constexpr int R = kDThreads / D4;
    // column sums over the row groups: every thread's partial float4 in
    // s_cols, then threads < d add the R partials of their column.
    static __device__ __forceinline__ void col_reduce(float4 part, float *s_cols, int rg, int col, int tid, int d,
                                                      float *dst) {
        *reinterpret_cast<float4 *>(s_cols + rg * d + col) = part;
        __syncthreads();
        if (tid < d) {
            float s = 0.f;
#pragma unroll
            for (int r2 = 0; r2 < R; ++r2) s += s_cols[r2 * d + tid];
            dst[tid] = s;
        }
        __syncthreads();
    }
};

// One delta-rule step on the thread's state rows; returns the thread's partial
// of q S (after the step) for its four columns.  s_w must hold w = k S.
template <int D4>
__device__ __forceinline__ float4 delta_rows(float4 (&st)[kDMaxRows], const float *s_k, const float *s_q,
                                             const float *s_v, const float *s_w, float alpha, float eb, int rg,
                                             int col, int c) {
    constexpr int R = kDThreads / D4;
    const float4 v4 = *reinterpret_cast<const float4 *>(s_v + col);
    const float4 w4 = *reinterpret_cast<const float4 *>(s_w + col);
    const float4 u = make_float4(v4.x - alpha * w4.x, v4.y - alpha * w4.y, v4.z - alpha * w4.z, v4.w - alpha * w4.w);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kDMaxRows; ++m) {
        const int r = rg + m * R;
        if (r < c) {
            const float kr = eb * s_k[r], qr = s_q[r];
            st[m].x = fmaf(alpha, st[m].x, kr * u.x);
            st[m].y = fmaf(alpha, st[m].y, kr * u.y);
            st[m].z = fmaf(alpha, st[m].z, kr * u.z);
            st[m].w = fmaf(alpha, st[m].w, kr * u.w);
            acc.x = fmaf(qr, st[m].x, acc.x);
            acc.y = fmaf(qr, st[m].y, acc.y);
            acc.z = fmaf(qr, st[m].z, acc.z);
            acc.w = fmaf(qr, st[m].w, acc.w);
        }
    }
    return acc;
}

// The thread's partial of w = k S for its four columns.
template <int D4>
__device__ __forceinline__ float4 key_answer(const float4 (&st)[kDMaxRows], const float *s_k, int rg, int c) {
    constexpr int R = kDThreads / D4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kDMaxRows; ++m) {
        const int r = rg + m * R;
        if (r < c) {
            const float kr = s_k[r];
            acc.x = fmaf(kr, st[m].x, acc.x);
            acc.y = fmaf(kr, st[m].y, acc.y);
            acc.z = fmaf(kr, st[m].z, acc.z);
            acc.w = fmaf(kr, st[m].w, acc.w);
        }
    }
    return acc;
}

// Two CTAs per SM (at most 128 registers a thread): the token-serial segments
// are many (one CTA each), so more of them run at once.
template <typename T, int D4>
__global__ void __launch_bounds__(kDThreads, 2)
delta_segment_kernel(DeltaArgs a, int32_t H, int32_t c, int32_t N, int32_t topk, int32_t use_shared, float scale) {
    constexpr int R = kDThreads / D4;
    constexpr int d = 4 * D4;
    extern __shared__ float smem[];
    float *s_k = smem, *s_q = s_k + c, *s_v = s_q + c, *s_w = s_v + d, *s_o = s_w + d, *s_cols = s_o + d;
    const T *q = static_cast<const T *>(a.q);
    const T *kk = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    const T *la = static_cast<const T *>(a.log_alpha);
    const T *bt = static_cast<const T *>(a.beta);
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
    const T *qsrc = is_shared && a.qs ? static_cast<const T *>(a.qs) : q;
    const T *ksrc = is_shared && a.ks ? static_cast<const T *>(a.ks) : kk;
    const int tid = threadIdx.x, cq = tid % D4, rg = tid / D4, col = 4 * cq;
    const int64_t state_off = (((int64_t)b * H + h) * P + slot) * (int64_t)c * d;
    // decode-style in-place use with nothing to do: leave the state alone
    if (len == 0 && a.init == a.final_state) return;

    float4 st[kDMaxRows];
#pragma unroll
    for (int m = 0; m < kDMaxRows; ++m) {
        const int r = rg + m * R;
        st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < c && a.init) st[m] = *reinterpret_cast<const float4 *>(a.init + state_off + (int64_t)r * d + col);
    }
    // row inputs travel one row ahead as raw elements
    struct Raw { T q, k, v, la, b; };
    auto fetch = [&](int n, int &t, int &jj, float &e) -> Raw {
        if (is_shared) {
            t = base + n;
            jj = 0;
            e = 1.f;
        } else {
            const int rec = a.perm_rec[base + n];
            t = rec / topk;
            jj = rec - t * topk;
            e = a.topk_w[((int64_t)t * H + h) * topk + jj];
        }
        const int64_t th = (int64_t)t * H + h;
        Raw x{};
        if (tid < c) {
            x.q = qsrc[th * c + tid];
            x.k = ksrc[th * c + tid];
        }
        if (tid < d) x.v = v[th * d + tid];
        x.la = la[th];
        x.b = bt[th];
        return x;
    };
    int t_nx = 0, j_nx = 0;
    float e_nx = 0.f;
    Raw x_nx{};
    if (len > 0) x_nx = fetch(0, t_nx, j_nx, e_nx);
    for (int n = 0; n < len; ++n) {
        const int t = t_nx, jj = j_nx;
        const float e = e_nx;
        const Raw x = x_nx;
        if (tid < c) {
            s_q[tid] = e * scale * to_f32(x.q);
            s_k[tid] = to_f32(x.k);
        }
        if (tid < d) s_v[tid] = to_f32(x.v);
        const float alpha = expf(to_f32(x.la)), eb = e * to_f32(x.b);
        if (n + 1 < len) x_nx = fetch(n + 1, t_nx, j_nx, e_nx);
        __syncthreads();
        DeltaRow<D4>::col_reduce(key_answer<D4>(st, s_k, rg, c), s_cols, rg, col, tid, d, s_w);
        DeltaRow<D4>::col_reduce(delta_rows<D4>(st, s_k, s_q, s_v, s_w, alpha, eb, rg, col, c), s_cols, rg, col,
                                 tid, d, s_o);
        const int64_t th = (int64_t)t * H + h;
        float *dst = is_shared ? a.part_shared + th * d : a.part_routed + (th * topk + jj) * d;
        if (tid < d) dst[tid] = s_o[tid];
    }
    if (a.final_state) {
#pragma unroll
        for (int m = 0; m < kDMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c) *reinterpret_cast<float4 *>(a.final_state + state_off + (int64_t)r * d + col) = st[m];
        }
    }
}

// Sum over the 16 lanes that share lane bit 4 of CB per-lane values (one per
// column), scattered: after halving steps on lane bits 3, 2, ... each lane
// holds one column's sum, column `owned` of the CB (from the lane's top bits),
// and the remaining steps add lanes that hold the same column -- both sides of
// every addition get the same operands, so the lanes agree bit for bit.
template <int CB>
__device__ __forceinline__ float reduce_scatter16(const float (&x)[CB], int rg, int &owned) {
    float a[CB];
#pragma unroll
    for (int j = 0; j < CB; ++j) a[j] = x[j];
    owned = 0;
#pragma unroll
    for (int m = 8, h = CB / 2; m >= 1; m >>= 1, h >>= 1) {
        if (h >= 1) {
            const bool hi = (rg & m) != 0;
#pragma unroll
            for (int j = 0; j < h; ++j) {
                const float send = hi ? a[j] : a[j + h];
                const float keep = hi ? a[j + h] : a[j];
                a[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
            owned += hi ? h : 0;
        } else {
            a[0] += __shfl_xor_sync(0xffffffffu, a[0], m);
        }
    }
    return a[0];
}

// Forward for c = 128 and d in {64, 128}: warp w holds columns
// [w d / 8, (w + 1) d / 8) of the state; lane (cg, rg) = (lane / 16, lane % 16)
// holds rows 8 rg .. 8 rg + 7 x CB = d / 16 columns from w d / 8 + cg CB.  A
// row then reads 8 k and 8 q values per thread from shared memory (k and q
// skewed by 4 floats per 32 rows, so that the 8 row groups of a quarter warp
// hit 8 distinct bank quads); the column sums w = k S and q S are register
// sums over the thread's 8 rows plus a reduce-scatter over the 16 row groups
// (lane shuffles), and u = e beta (v - alpha w) goes back to the warp's lanes
// through a per-warp shared buffer.  Column pairs go through the packed
// float32 pipe (each lane the scalar operation).
//
// One CTA barrier per row: the next row's q, k and v are written into the
// other half of a double buffer right after it, while the three rows after
// that are in flight in registers (the loop is unrolled by three so that no
// register slot is copied while its loads are pending).  A routed item's
// records come in blocks of 32 rows through shared memory (warp 0 loads block
// m + 1 at row 32 m and stores it at row 32 m + 16), so that no row's input
// loads wait on its record.
//
// Measured on the layer shape (8 x 4096 tokens, H16, N8, top-2, shared):
// 8.45 ms against 10.7 ms for delta_segment_kernel.  The kernel issues on
// about 45 % of cycles with two warps per scheduler, stalled mostly on
// fixed-latency dependencies; neither half-width CTAs at two per SM, nor a
// recurrence arranged to take the reduction off the row-to-row path (w_{n+1}
// = alpha_n k_{n+1} S_{n-1} + (k_{n+1} . k_n) u_n), nor scalar instead of
// packed arithmetic was faster (9.5 - 10.0 ms).
template <typename T, int D>
__global__ void __launch_bounds__(kDThreads, 1)
delta_cols_kernel(DeltaArgs a, int32_t H, int32_t N, int32_t topk, int32_t use_shared, float scale) {
    constexpr int C = 128, CB = D / 16, CP = CB / 2, WC = D / 8;
    constexpr int CS = C + C / 8;  // skewed k / q row
    __shared__ __align__(16) float s_k[2][CS], s_q[2][CS], s_v[2][D];
    __shared__ __align__(16) float s_u[8][2][WC];  // per warp, by row parity
    __shared__ float s_sc[2][3];                   // alpha, e * beta, e * scale of the row
    __shared__ int64_t s_dst[2];                   // first element of the row's read-out slot
    __shared__ int s_rec[2][32];                   // records of rows 32 m .. 32 m + 31 in s_rec[m % 2]
    const T *q = static_cast<const T *>(a.q);
    const T *kk = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    const T *la = static_cast<const T *>(a.log_alpha);
    const T *bt = static_cast<const T *>(a.beta);
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
    const T *qsrc = is_shared && a.qs ? static_cast<const T *>(a.qs) : q;
    const T *ksrc = is_shared && a.ks ? static_cast<const T *>(a.ks) : kk;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rg = lane & 15, cg = lane >> 4;
    const int col0 = warp * WC + cg * CB;     // first of the thread's CB columns
    const int kofs = 8 * rg + 4 * (rg >> 2);  // its 8 rows in the skewed k / q rows
    const int64_t state_off = (((int64_t)b * H + h) * P + slot) * (int64_t)C * D;
    if (len == 0 && a.init == a.final_state) return;
    F2 st[8][CP];  // rows 8 rg + i, column pairs from col0
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int j4 = 0; j4 < CB / 4; ++j4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (a.init) x = *reinterpret_cast<const float4 *>(a.init + state_off + (int64_t)(8 * rg + i) * D + col0 + 4 * j4);
            st[i][2 * j4] = f2(x.x, x.y);
            st[i][2 * j4 + 1] = f2(x.z, x.w);
        }
    }
    // one row's inputs as raw elements: q, k (threads < c), v (threads < d)
    struct Raw { T q, k, v, la, b; float e; int64_t dst; };
    auto fetch = [&](int n) -> Raw {
        int t, jj;
        Raw x{};
        if (is_shared) {
            t = base + n;
            jj = 0;
            x.e = 1.f;
        } else {
            const int rec = s_rec[(n >> 5) & 1][n & 31];
            t = rec / topk;
            jj = rec - t * topk;
            x.e = a.topk_w[((int64_t)t * H + h) * topk + jj];
        }
        const int64_t th = (int64_t)t * H + h;
        if (tid < C) {
            x.q = qsrc[th * C + tid];
            x.k = ksrc[th * C + tid];
        }
        if (tid < D) x.v = v[th * D + tid];
        x.la = la[th];
        x.b = bt[th];
        x.dst = is_shared ? th * D : (th * topk + jj) * D;
        return x;
    };
    auto put = [&](const Raw &x, int buf) {
        if (tid < C) {
            const int r = tid + 4 * (tid >> 5);
            s_q[buf][r] = to_f32(x.q);
            s_k[buf][r] = to_f32(x.k);
        }
        if (tid < D) s_v[buf][tid] = to_f32(x.v);
        if (tid == 0) {
            s_sc[buf][0] = expf(to_f32(x.la));
            s_sc[buf][1] = x.e * to_f32(x.b);
            s_sc[buf][2] = x.e * scale;
            s_dst[buf] = x.dst;
        }
    };
    float *out = is_shared ? a.part_shared : a.part_routed;
    int rec_next = 0;
    if (!is_shared && tid < 32) {
        if (tid < len) s_rec[0][tid] = a.perm_rec[base + tid];
    }
    __syncthreads();
    auto compute = [&](int cb) {
        const float *kb = s_k[cb] + kofs, *qb = s_q[cb] + kofs;
        const float alpha = s_sc[cb][0], eb = s_sc[cb][1], qf = s_sc[cb][2];
        const float4 ka = *reinterpret_cast<const float4 *>(kb), kz = *reinterpret_cast<const float4 *>(kb + 4);
        const float kr[8] = {ka.x, ka.y, ka.z, ka.w, kz.x, kz.y, kz.z, kz.w};
        F2 wp[CP];
#pragma unroll
        for (int j = 0; j < CP; ++j) wp[j] = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const F2 k2 = f2(kr[i], kr[i]);
#pragma unroll
            for (int j = 0; j < CP; ++j) wp[j] = fma2(k2, st[i][j], wp[j]);
        }
        float wl[CB];
#pragma unroll
        for (int j = 0; j < CP; ++j) {
            const float2 x = f2_get(wp[j]);
            wl[2 * j] = x.x;
            wl[2 * j + 1] = x.y;
        }
        int own;
        const float w = reduce_scatter16<CB>(wl, rg, own);
        // u of the owned column, to every lane of the column group
        float *su = s_u[warp][cb];
        if ((rg & (16 / CB - 1)) == 0) su[cg * CB + own] = eb * (s_v[cb][col0 + own] - alpha * w);
        __syncwarp();
        F2 u2[CP];
#pragma unroll
        for (int j4 = 0; j4 < CB / 4; ++j4) {
            const float4 x = *reinterpret_cast<const float4 *>(su + cg * CB + 4 * j4);
            u2[2 * j4] = f2(x.x, x.y);
            u2[2 * j4 + 1] = f2(x.z, x.w);
        }
        const float4 qa = *reinterpret_cast<const float4 *>(qb), qz = *reinterpret_cast<const float4 *>(qb + 4);
        const float qr[8] = {qa.x, qa.y, qa.z, qa.w, qz.x, qz.y, qz.z, qz.w};
        // S <- alpha S + k u, then the read-out q S after the step
        const F2 a2 = f2(alpha, alpha);
#pragma unroll
        for (int j = 0; j < CP; ++j) wp[j] = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const F2 k2 = f2(kr[i], kr[i]), q2 = f2(qr[i], qr[i]);
#pragma unroll
            for (int j = 0; j < CP; ++j) {
                st[i][j] = fma2(k2, u2[j], mul2(a2, st[i][j]));
                wp[j] = fma2(q2, st[i][j], wp[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < CP; ++j) {
            const float2 x = f2_get(wp[j]);
            wl[2 * j] = x.x;
            wl[2 * j + 1] = x.y;
        }
        const float o = reduce_scatter16<CB>(wl, rg, own);
        if ((rg & (16 / CB - 1)) == 0) out[s_dst[cb] + col0 + own] = qf * o;
    };
    auto step = [&](int n, Raw &slot) {
        const int cb = n & 1;
        // row n's buffer is complete; every thread has finished row n - 1,
        // which read the other buffer
        __syncthreads();
        if (!is_shared && tid < 32) {
            const int nb = n + 32 - (n & 31) + tid;  // row tid of the next block
            if ((n & 31) == 0 && nb < len) rec_next = a.perm_rec[base + nb];
            if ((n & 31) == 16 && nb < len) s_rec[((n >> 5) + 1) & 1][tid] = rec_next;
        }
        if (n + 1 < len) {
            put(slot, cb ^ 1);
            if (n + 4 < len) slot = fetch(n + 4);
        }
        compute(cb);
    };
    Raw ra{}, rb{}, rc{};
    if (len > 0) put(fetch(0), 0);
    if (len > 1) ra = fetch(1);
    if (len > 2) rb = fetch(2);
    if (len > 3) rc = fetch(3);
    for (int n = 0; n < len; n += 3) {
        step(n, ra);
        if (n + 1 < len) step(n + 1, rb);
        if (n + 2 < len) step(n + 2, rc);
    }
    if (a.final_state) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int j4 = 0; j4 < CB / 4; ++j4) {
                const float2 lo = f2_get(st[i][2 * j4]), hi = f2_get(st[i][2 * j4 + 1]);
                *reinterpret_cast<float4 *>(a.final_state + state_off + (int64_t)(8 * rg + i) * D + col0 + 4 * j4) =
                    make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
    }
}

// Decode: one CTA per (sequence, head).
// Two CTAs per SM (at most 128 registers a thread): each holds one state in
// registers between its load and its store, so the second CTA keeps HBM busy
// through the first one's reductions.
template <typename T, int D4>
__global__ void __launch_bounds__(kDThreads, 2)
delta_decode_kernel(DeltaDecodeArgs a, int32_t H, int32_t c, int32_t N, int32_t topk, int32_t use_shared,
                    float scale) {
    constexpr int R = kDThreads / D4;
    constexpr int d = 4 * D4;
    extern __shared__ float smem[];
    float *s_k = smem, *s_q = s_k + c, *s_v = s_q + c, *s_w = s_v + d, *s_o = s_w + d, *s_cols = s_o + d;
    __shared__ int s_idx[kMaxTopK];
    __shared__ float s_e[kMaxTopK];
    const int bh = blockIdx.x;
    const int tid = threadIdx.x, cq = tid % D4, rg = tid / D4, col = 4 * cq;
    const int P = N + use_shared;
    if (tid < 32) {
        int idx[kMaxTopK];
        float w[kMaxTopK];
        route_token_warp<T>(static_cast<const T *>(a.logits) + (int64_t)bh * N, N, topk, tid, idx, w);
        if (tid == 0) {
            for (int j = 0; j < topk; ++j) {
                s_idx[j] = idx[j];
                s_e[j] = w[j];
                if (a.topk_idx) a.topk_idx[(int64_t)bh * topk + j] = idx[j];
                if (a.topk_w) a.topk_w[(int64_t)bh * topk + j] = w[j];
            }
        }
    }
    const float alpha = expf(to_f32(static_cast<const T *>(a.log_alpha)[bh]));
    const float beta = to_f32(static_cast<const T *>(a.beta)[bh]);
    float o_col = 0.f;  // thread tid < d: column tid of the output
    for (int j = 0; j < topk + use_shared; ++j) {
        __syncthreads();  // routing written; the previous slot's shared memory consumed
        const bool shared_slot = j == topk;
        const int slot = shared_slot ? N : s_idx[j];
        const float e = shared_slot ? 1.f : s_e[j];
        const T *qsrc = static_cast<const T *>(shared_slot && a.qs ? a.qs : a.q);
        const T *ksrc = static_cast<const T *>(shared_slot && a.ks ? a.ks : a.k);
        if (tid < c) {
            s_q[tid] = e * scale * to_f32(qsrc[(int64_t)bh * c + tid]);
            s_k[tid] = to_f32(ksrc[(int64_t)bh * c + tid]);
        }
        if (tid < d) s_v[tid] = to_f32(static_cast<const T *>(a.v)[(int64_t)bh * d + tid]);
        float *S = a.state + ((int64_t)bh * P + slot) * (int64_t)c * d;
        float4 st[kDMaxRows];
#pragma unroll
        for (int m = 0; m < kDMaxRows; ++m) {
            const int r = rg + m * R;
            st[m] = r < c ? __ldcs(reinterpret_cast<const float4 *>(S + (int64_t)r * d + col))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        DeltaRow<D4>::col_reduce(key_answer<D4>(st, s_k, rg, c), s_cols, rg, col, tid, d, s_w);
        DeltaRow<D4>::col_reduce(delta_rows<D4>(st, s_k, s_q, s_v, s_w, alpha, e * beta, rg, col, c), s_cols, rg,
                                 col, tid, d, s_o);
        if (tid < d) o_col += s_o[tid];
#pragma unroll
        for (int m = 0; m < kDMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c) __stcs(reinterpret_cast<float4 *>(S + (int64_t)r * d + col), st[m]);
        }
    }
    if (tid < d) Elem<T>::store(static_cast<T *>(a.out) + (int64_t)bh * d + tid, o_col);
}

template <typename T, int D4>
cudaError_t launch_fwd_t(const sse_config_t &cfg, const DeltaArgs &a, cudaStream_t stream) {
    constexpr int R = kDThreads / D4;
    const int c = cfg.key_dim, d = 4 * D4;
    const size_t smem = sizeof(float) * (2 * c + 3 * d + R * d);
    const int64_t nseg = (int64_t)a.num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    if (nseg == 0) return cudaSuccess;
    if constexpr (4 * D4 == 64 || 4 * D4 == 128) {
        if (c == 128) {
            delta_cols_kernel<T, 4 * D4><<<(unsigned)nseg, kDThreads, 0, stream>>>(
                a, cfg.num_heads, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale);
            return cudaGetLastError();
        }
    }
    delta_segment_kernel<T, D4><<<(unsigned)nseg, kDThreads, smem, stream>>>(
        a, cfg.num_heads, c, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale);
    return cudaGetLastError();
}

template <typename T, int D4>
cudaError_t launch_dec_t(const sse_config_t &cfg, const DeltaDecodeArgs &a, cudaStream_t stream) {
    constexpr int R = kDThreads / D4;
    const int c = cfg.key_dim, d = 4 * D4;
    const size_t smem = sizeof(float) * (2 * c + 3 * d + R * d);
    const int64_t rows = (int64_t)a.batch * cfg.num_heads;
    if (rows == 0) return cudaSuccess;
    delta_decode_kernel<T, D4><<<(unsigned)rows, kDThreads, smem, stream>>>(
        a, cfg.num_heads, c, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale);
    return cudaGetLastError();
}

template <typename T, typename Args, cudaError_t (*F16)(const sse_config_t &, const Args &, cudaStream_t),
          cudaError_t (*F32)(const sse_config_t &, const Args &, cudaStream_t),
          cudaError_t (*F64)(const sse_config_t &, const Args &, cudaStream_t),
          cudaError_t (*F128)(const sse_config_t &, const Args &, cudaStream_t),
          cudaError_t (*F256)(const sse_config_t &, const Args &, cudaStream_t)>
cudaError_t by_d(const sse_config_t &cfg, const Args &a, cudaStream_t stream) {
    switch (cfg.value_dim) {
    case 16: return F16(cfg, a, stream);
    case 32: return F32(cfg, a, stream);
    case 64: return F64(cfg, a, stream);
    case 128: return F128(cfg, a, stream);
    case 256: return F256(cfg, a, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t fwd_dispatch(const sse_config_t &cfg, const DeltaArgs &a, cudaStream_t stream) {
    return by_d<T, DeltaArgs, launch_fwd_t<T, 4>, launch_fwd_t<T, 8>, launch_fwd_t<T, 16>, launch_fwd_t<T, 32>,
                launch_fwd_t<T, 64>>(cfg, a, stream);
}

template <typename T>
cudaError_t dec_dispatch(const sse_config_t &cfg, const DeltaDecodeArgs &a, cudaStream_t stream) {
    return by_d<T, DeltaDecodeArgs, launch_dec_t<T, 4>, launch_dec_t<T, 8>, launch_dec_t<T, 16>, launch_dec_t<T, 32>,
                launch_dec_t<T, 64>>(cfg, a, stream);
}

}  // namespace

bool delta_supported(const sse_config_t &cfg) {
    const int d = cfg.value_dim, c = cfg.key_dim;
    if (!(d == 16 || d == 32 || d == 64 || d == 128 || d == 256)) return false;
    const int R = kDThreads / (d / 4);
    return c >= 1 && c <= R * kDMaxRows && c <= kDThreads;
}

// The chunked tensor-core form (delta_chunked.cu) unless the token-serial one
// is asked for (SSE_ALGO_RECURRENT) or the shape has no chunked form.
cudaError_t launch_delta_forward(const sse_config_t &cfg, const DeltaArgs &a, cudaStream_t stream) {
    if (delta_chunked_partials_bf16(cfg)) return launch_delta_chunked(cfg, a, stream);
    return cfg.dtype == SSE_BF16 ? fwd_dispatch<__nv_bfloat16>(cfg, a, stream) : fwd_dispatch<float>(cfg, a, stream);
}

cudaError_t launch_delta_decode(const sse_config_t &cfg, const DeltaDecodeArgs &a, cudaStream_t stream) {
    return cfg.dtype == SSE_BF16 ? dec_dispatch<__nv_bfloat16>(cfg, a, stream) : dec_dispatch<float>(cfg, a, stream);
}

}  // namespace sse
