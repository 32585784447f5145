// softmax.cuh -- row softmax / log-softmax (forward, backward) and per-row cross-entropy
// (forward, backward) on the row skeleton of the normalization kernels.
//
// Sources (page title, section): tensorcore "Training kernels", "Softmax -- standalone,
// row-wise" (subtract the row maximum, exponentiate, sum, divide; backward from Y and
// dY); meTile "Kernel coverage and training scope", the reduction and loss checklists
// (softmax / log-softmax with input gradients; cross-entropy with integer targets, an
// index whose rows are skipped, losses left per row or summed or averaged, label
// smoothing spread evenly over the classes, a penalty on the squared log-sum-exp, and
// the maxima and log-denominators kept for the backward); "Metal subgroup
// LayerNorm and cross-entropy report", "Structural repair exercised by cross-entropy"
// (loss = log(total) + peak - selected).
//
//  * Softmax keeps the row in registers like the normalization forward (two row
//    reductions: the maximum, then the sum of exp(x - max)); its backward keeps Y and dY
//    (one reduction: sum dY*Y, or sum dY for log-softmax). Neither has parameters, so
//    neither has partials: one row group per row, non-persistent.
//  * Cross-entropy rows may be far wider than registers hold (vocabularies), so the
//    forward streams each row once, keeping a running maximum and a running sum of
//    exp(x - running max) (rescaled when the maximum grows), the sum of x (for label
//    smoothing), and reads the target logit directly; the per-thread states combine
//    with the same rescaling in a fixed order. The backward streams the row again and
//    needs no reduction: dX = g * ((1 + 2 z lse) exp(x - lse) - q). A last small kernel
//    sums the per-row losses in a fixed order for the sum/mean reductions.
//  * exp is __expf (the hardware exp2 path): relative error about 2^-21 for the ranges
//    met here, well inside every output tolerance; log is logf, once per row. The
//    cross-entropy loops, which are instruction-bound, write exp(x - m) as
//    2^(x log2(e) - m log2(e)): one fp32x2 fused multiply-add for two arguments, then
//    the hardware base-2 exponential (ex2.approx, relative error about 2^-22); the
//    rounding of m log2(e) adds about |m| 2^-24 to the exponent.
#pragma once

#include "kernels.cuh"

namespace mt {

struct SoftmaxArgs {
    const void *X;   // forward: X; backward: the forward output Y
    const void *dY;  // backward only
    void *Y;         // forward: Y; backward: dX
    int64_t N;
    int D;
    int xdt, gdt;    // storage types (scalar fallback): X/Y/dX, and dY
    int slice;       // cluster-split streaming kernels: columns per CTA (a multiple of 8)
};

struct CeArgs {
    const void *X;             // logits [N, D]
    const int64_t *T;          // targets [N]
    float *loss;               // forward: per-row loss [N]
    float *lse;                // forward: written; backward: read [N]
    const float *dloss;        // backward: [N] (none) or [1] (sum, mean)
    const float *n_valid;      // backward, mean: the forward's count of valid rows
    void *dX;                  // backward: [N, D]
    int64_t N;
    int D;
    int64_t ignore_index;
    float eps;                 // label smoothing
    float z;                   // z-loss coefficient
    int reduction;             // 0 none, 1 sum, 2 mean
    int xdt;                   // storage type of X and dX (scalar fallback)
};

// Maximum over the TPR threads of one row group (same pattern as row_sum, fmaxf).
template <int TPR, int RPC>
__device__ __forceinline__ float row_max(float v, float *red, int buf, int rg, int wir, int lane) {
    constexpr int WPR = TPR / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (WPR > 1) {
        float *s = red + (buf * RPC + rg) * WPR;
        if (lane == 0) s[wir] = v;
        row_group_sync<TPR, RPC, false>(rg);
        v = lane < WPR ? s[lane] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    }
    return v;
}

// ------------------------------------------------------------------ softmax ---

// Forward for aligned rows (D % 8 == 0): one row group of TPR threads per row, thread t
// owning CH chunks of 8 at columns (k*TPR + t)*8; the row stays in fp32 pairs.
template <int TPR, int RPC, int CH, bool LOG, int XT>
__global__ void __launch_bounds__(TPR * RPC)
softmax_fwd_vec8_kernel(const SoftmaxArgs a) {
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * RPC * WPR];
    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const int64_t row = (int64_t)blockIdx.x * RPC + rg;
    const bool ok = row < a.N;
    if (ok) prefetch_l2_row<TPR, CH>(as<XT>(a.X) + row * (int64_t)D, D, t);
    pdl_enter();
    if (WPR == 1 && !ok) return;
    const int64_t off = (ok ? row : 0) * (int64_t)D;

    float2 x[CH][4];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        const bool v = ok && col < D;
        ld_chunk<XT, kStream>(as<XT>(a.X) + off + col, v, x[k]);
        if (v) {
#pragma unroll
            for (int p = 0; p < 4; ++p) m = fmaxf(m, fmaxf(x[k][p].x, x[k][p].y));
        }
    }
    m = row_max<TPR, RPC>(m, red, 0, rg, wir, lane);
    float s[1] = {0.f};
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        if (!(ok && (k * TPR + t) * 8 < D)) continue;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            x[k][p] = make_float2(x[k][p].x - m, x[k][p].y - m);
            if constexpr (!LOG) x[k][p] = make_float2(__expf(x[k][p].x), __expf(x[k][p].y));
            s[0] += LOG ? (__expf(x[k][p].x) + __expf(x[k][p].y)) : (x[k][p].x + x[k][p].y);
        }
    }
    row_sum<TPR, RPC, 1>(s, red, 1, rg, wir, lane);
    if (!ok) return;
    const float inv = 1.0f / s[0], ls = logf(s[0]);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        if (col >= D) continue;
        float2 y[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            y[p] = LOG ? make_float2(x[k][p].x - ls, x[k][p].y - ls)
                       : make_float2(x[k][p].x * inv, x[k][p].y * inv);
        st_chunk<XT>(as<XT>(a.Y) + off + col, y);
    }
}

// Backward for aligned rows from the forward output Y (type XT) and dY (type XT):
//   softmax: dX = Y * (dY - sum dY*Y);  log-softmax: dX = dY - exp(Y) * sum dY.
template <int TPR, int RPC, int CH, bool LOG, int XT>
__global__ void __launch_bounds__(TPR * RPC)
softmax_bwd_vec8_kernel(const SoftmaxArgs a) {
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * RPC * WPR];
    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const int64_t row = (int64_t)blockIdx.x * RPC + rg;
    const bool ok = row < a.N;
    if (ok) {
        prefetch_l2_row<TPR, CH>(as<XT>(a.X) + row * (int64_t)D, D, t);
        prefetch_l2_row<TPR, CH>(as<XT>(a.dY) + row * (int64_t)D, D, t);
    }
    pdl_enter();
    if (WPR == 1 && !ok) return;
    const int64_t off = (ok ? row : 0) * (int64_t)D;

    float2 y[CH][4], dy[CH][4];
    float dot[1] = {0.f};
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        const bool v = ok && col < D;
        ld_chunk<XT, kStream>(as<XT>(a.X) + off + col, v, y[k]);
        ld_chunk<XT, kStream>(as<XT>(a.dY) + off + col, v, dy[k]);
#pragma unroll
        for (int p = 0; p < 4; ++p)
            dot[0] += LOG ? (dy[k][p].x + dy[k][p].y) : (dy[k][p].x * y[k][p].x + dy[k][p].y * y[k][p].y);
    }
    row_sum<TPR, RPC, 1>(dot, red, 0, rg, wir, lane);
    if (!ok) return;
    const float c = dot[0];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        if (col >= D) continue;
        float2 o[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            o[p] = LOG ? make_float2(dy[k][p].x - __expf(y[k][p].x) * c, dy[k][p].y - __expf(y[k][p].y) * c)
                       : make_float2(y[k][p].x * (dy[k][p].x - c), y[k][p].y * (dy[k][p].y - c));
        st_chunk<XT>(as<XT>(a.Y) + off + col, o);
    }
}

// Scalar forward/backward for any alignment and width (types at run time): thread t of a
// row group owns columns k*TPR + t, k < CH.
template <int TPR, int RPC, int CH, bool LOG, bool BWD>
__global__ void __launch_bounds__(TPR * RPC, 1)
softmax_scalar_kernel(const SoftmaxArgs a) {
    pdl_enter();
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * RPC * WPR];
    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const int64_t row = (int64_t)blockIdx.x * RPC + rg;
    const bool ok = row < a.N;
    if (WPR == 1 && !ok) return;
    const int64_t off = (ok ? row : 0) * (int64_t)D;
    const int lim = ok ? D : 0;

    float x[CH], dy[BWD ? CH : 1];
    if constexpr (!BWD) {
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = k * TPR + t;
            x[k] = col < lim ? ld_elem_stream(a.X, off + col, a.xdt) : -INFINITY;
            m = fmaxf(m, x[k]);
        }
        m = row_max<TPR, RPC>(m, red, 0, rg, wir, lane);
        float s[1] = {0.f};
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            if (k * TPR + t >= lim) continue;
            x[k] -= m;
            s[0] += __expf(x[k]);
        }
        row_sum<TPR, RPC, 1>(s, red, 1, rg, wir, lane);
        if (!ok) return;
        const float inv = 1.0f / s[0], ls = logf(s[0]);
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = k * TPR + t;
            if (col >= D) continue;
            st_elem(a.Y, off + col, LOG ? x[k] - ls : __expf(x[k]) * inv, a.xdt);
        }
    } else {
        float dot[1] = {0.f};
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = k * TPR + t;
            const bool v = col < lim;
            x[k] = v ? ld_elem_stream(a.X, off + col, a.xdt) : 0.f;
            dy[k] = v ? ld_elem_stream(a.dY, off + col, a.gdt) : 0.f;
            dot[0] += LOG ? dy[k] : dy[k] * x[k];
        }
        row_sum<TPR, RPC, 1>(dot, red, 0, rg, wir, lane);
        if (!ok) return;
        const float c = dot[0];
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = k * TPR + t;
            if (col >= D) continue;
            st_elem(a.Y, off + col, LOG ? dy[k] - __expf(x[k]) * c : x[k] * (dy[k] - c), a.xdt);
        }
    }
}

// ------------------------------------------------------------- cross-entropy ---

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)

// 2^x by the hardware's approximate base-2 exponential (subnormal results flush to 0,
// 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Each cross-entropy thread loads UN chunks (a kernel template parameter, set per shape)
// before using the first: the bytes in flight.

// Running (maximum, sum of exp(x - maximum)) state and its order-fixed combination. A
// state whose maximum is -inf has seen only -inf logits (masked columns) and sums to 0.
struct MaxSum {
    float m, s;
};
__device__ __forceinline__ MaxSum combine(MaxSum a, MaxSum b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    return {m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}
__device__ __forceinline__ void add_value(MaxSum &st, float x) {
    if (x > st.m) {
        st.s = st.s * __expf(st.m - x) + 1.f;
        st.m = x;
    } else if (st.m != -INFINITY) {
        st.s += __expf(x - st.m);
    }
}

// Loads the UN chunks c0, c0 + TPR, ... of one row (zeros past the end).
template <int TPR, int XT, int UN>
__device__ __forceinline__ void ce_load(const void *X, int64_t off, int c0, int D,
                                        float2 (&f)[UN][4]) {
#pragma unroll
    for (int u = 0; u < UN; ++u) {
        const int c = c0 + u * TPR;
        ld_chunk<XT, kStream>(as<XT>(X) + off + c * 8, c * 8 < D, f[u]);
    }
}

// The 16-byte units of the UN chunks c0, c0 + TPR, ... of one row, as loaded; chunks
// past the end read as -inf (they must not raise the running maximum).
template <int TPR, int XT, int UN, int H = kStream>
__device__ __forceinline__ void ce_load_raw(const void *X, int64_t off, int c0, int D,
                                            uint4 (&raw)[UN][chunk_units<XT>()]) {
    constexpr uint32_t kNegInf = (XT == kF32) ? 0xff800000u : (XT == kBF16) ? 0xff80ff80u : 0xfc00fc00u;
#pragma unroll
    for (int u = 0; u < UN; ++u) {
        const int c = c0 + u * TPR;
#pragma unroll
        for (int q = 0; q < chunk_units<XT>(); ++q)
            raw[u][q] = c * 8 < D ? ld_unit<H>(as<XT>(X) + off + c * 8 + q * (8 / chunk_units<XT>()))
                                  : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
    }
}

// Maximum of one loaded chunk: 2-byte types with packed two-lane max instructions on the
// loaded words (a maximum is exact, so this equals the fp32 maximum of the widened
// values), fp32 lane by lane.
template <int XT>
__device__ __forceinline__ float chunk_max(const uint4 (&r)[chunk_units<XT>()]) {
    if constexpr (XT == kF32) {
        float m = -INFINITY;
#pragma unroll
        for (int q = 0; q < chunk_units<XT>(); ++q)
            m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(r[q].x), __uint_as_float(r[q].y)),
                               fmaxf(__uint_as_float(r[q].z), __uint_as_float(r[q].w))));
        return m;
    } else if constexpr (XT == kBF16) {
        auto w = [](uint32_t v) { return *reinterpret_cast<const __nv_bfloat162 *>(&v); };
        const __nv_bfloat162 m = __hmax2(__hmax2(w(r[0].x), w(r[0].y)), __hmax2(w(r[0].z), w(r[0].w)));
        return __bfloat162float(__hmax(m.x, m.y));
    } else {
        auto w = [](uint32_t v) { return *reinterpret_cast<const __half2 *>(&v); };
        const __half2 m = __hmax2(__hmax2(w(r[0].x), w(r[0].y)), __hmax2(w(r[0].z), w(r[0].w)));
        return __half2float(__hmax(m.x, m.y));
    }
}

// Element e (0..7) of an 8-element chunk held as four fp32 pairs.
__device__ __forceinline__ float chunk_elem(const float2 (&f)[4], int e) {
    float v = f[0].x;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        v = (e == 2 * p) ? f[p].x : v;
        v = (e == 2 * p + 1) ? f[p].y : v;
    }
    return v;
}

// A row group of TPR threads per row: one CTA per row, or, with one warp per row, RPC
// rows (warps) per CTA. VEC8: 8-element chunks (D % 8 == 0, aligned rows), thread t
// taking chunks t, t + TPR, ...; otherwise single elements, same striding. Every thread
// reads the row's target with its first logits; the thread that meets the target column
// keeps its logit, so no load waits on another at the end of the row.
template <int TPR, int RPC, bool VEC8, int XT, int MINB, int UN>
__global__ void __launch_bounds__(TPR * RPC, MINB)
ce_fwd_kernel(const CeArgs a) {
    constexpr int W = TPR / 32;
    static_assert(W <= 32 && (W & (W - 1)) == 0, "warps per row: a power of two up to 32");
    static_assert(W == 1 || RPC == 1, "several rows per CTA only with a warp per row");
    __shared__ float sm_m[W], sm_s[W], sm_x[W], sm_t[RPC];
    const int tid = threadIdx.x, t = tid % TPR, rg = tid / TPR, lane = tid % 32, w = t / 32;
    const int64_t row = (int64_t)blockIdx.x * RPC + rg;
    // the first batch of UN chunks a thread (aligned rows only: the scalar form's XT
    // stands for a type read at run time)
    if (VEC8 && row < a.N) prefetch_l2(as<XT>(a.X) + row * (int64_t)a.D, min(a.D, UN * TPR * 8), t, TPR);
    pdl_enter();
    if (RPC > 1 && row >= a.N) return;  // a warp-wide row group: no CTA barrier below
    const int D = a.D;
    const int64_t off = row * (int64_t)D;

    MaxSum st{-INFINITY, 0.f};
    float sx = 0.f;
    if constexpr (VEC8) {
        // per batch of UN chunks: one running-maximum update (from the chunks'
        // packed maxima), then the exponentials of the valid chunks
        constexpr int CU = chunk_units<XT>();
        const float2 l2e = make_float2(kLog2e, kLog2e);
        float2 sx2 = make_float2(0.f, 0.f);
        uint4 raw[UN][CU];
        ce_load_raw<TPR, XT, UN>(a.X, off, t, D, raw);
        const int64_t tg = a.T[row];
        const int tc = (tg >= 0 && tg < D) ? (int)(tg >> 3) : -1;   // chunk holding the target
        for (int c0 = t;;) {
            float bm = chunk_max<XT>(raw[0]);
#pragma unroll
            for (int u = 1; u < UN; ++u) bm = fmaxf(bm, chunk_max<XT>(raw[u]));
            const float m = fmaxf(st.m, bm);
            const float ms = (m == -INFINITY) ? 0.f : m;   // all -inf so far: exps are 0
            const float nb = -ms * kLog2e;
            const float2 nb2 = make_float2(nb, nb);
            st.s *= ex2(fmaf(st.m, kLog2e, nb));
            st.m = m;
            float2 cs2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                const int c = c0 + u * TPR;
                if (c * 8 >= D) continue;
                float2 f[4];
                unpack_chunk<XT, 4>(raw[u], 1, f);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 e = __ffma2_rn(f[p], l2e, nb2);   // (x - ms) log2(e)
                    cs2 = __fadd2_rn(cs2, make_float2(ex2(e.x), ex2(e.y)));
                    sx2 = __fadd2_rn(sx2, f[p]);
                }
                if (c == tc) sm_t[rg] = chunk_elem(f, (int)(tg & 7));
            }
            st.s += cs2.x + cs2.y;
            c0 += UN * TPR;
            if (c0 * 8 >= D) break;
            ce_load_raw<TPR, XT, UN>(a.X, off, c0, D, raw);
        }
        sx = sx2.x + sx2.y;
    } else {
        const int64_t tg = a.T[row];
        for (int j = t; j < D; j += TPR) {
            const float v = ld_elem_stream(a.X, off + j, a.xdt);
            add_value(st, v);
            sx += v;
            if (j == tg) sm_t[rg] = v;
        }
    }
    // fixed-order combination: butterfly within each warp, then across the W warp results
    // (lower-indexed partial first in every pair)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum other{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.s, o)};
        st = (lane & o) ? combine(other, st) : combine(st, other);
        sx += __shfl_xor_sync(0xffffffffu, sx, o);
    }
    MaxSum tot = st;
    float tx = sx;
    if constexpr (W == 1) {
        __syncwarp();  // the target logit's owner wrote sm_t[rg]
    } else {
        if (lane == 0) {
            sm_m[w] = st.m;
            sm_s[w] = st.s;
            sm_x[w] = sx;
        }
        __syncthreads();
        if (w != 0) return;
        tot = MaxSum{lane < W ? sm_m[lane] : -INFINITY, lane < W ? sm_s[lane] : 0.f};
        tx = lane < W ? sm_x[lane] : 0.f;
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) {
            MaxSum other{__shfl_xor_sync(0xffffffffu, tot.m, o), __shfl_xor_sync(0xffffffffu, tot.s, o)};
            tot = (lane & o) ? combine(other, tot) : combine(tot, other);
            tx += __shfl_xor_sync(0xffffffffu, tx, o);
        }
    }
    if (lane == 0) {
        const float l = tot.m + logf(tot.s);
        a.lse[row] = l;
        const int64_t tg = a.T[row];
        float loss;
        if (tg == a.ignore_index) {
            loss = 0.f;
        } else if (tg < 0 || tg >= D) {
            loss = __int_as_float(0x7fc00000);
        } else {
            loss = l - (1.f - a.eps) * sm_t[rg] - (a.eps / (float)D) * tx + a.z * l * l;
        }
        a.loss[row] = loss;
    }
}

// The upstream gradient of a row whose target is tg (0 for an ignored row). The loads
// do not wait on tg, so they are issued together.
__device__ __forceinline__ float ce_row_grad(const CeArgs &a, int64_t row, int64_t tg) {
    const float d = a.dloss[a.reduction == 0 ? row : 0];
    const float n = (a.reduction == 2) ? a.n_valid[0] : 1.f;
    float g = (a.reduction == 2) ? (n > 0.f ? d / n : 0.f) : d;
    return tg == a.ignore_index ? 0.f : g;
}

template <int TPR, int RPC, bool VEC8, int XT, int MINB, int UN>
__global__ void __launch_bounds__(TPR * RPC, MINB)
ce_bwd_kernel(const CeArgs a) {
    const int t = threadIdx.x % TPR;
    const int64_t row = (int64_t)blockIdx.x * RPC + threadIdx.x / TPR;
    // the first batch of UN chunks a thread (aligned rows only: the scalar form's XT
    // stands for a type read at run time)
    if (VEC8 && row < a.N) prefetch_l2(as<XT>(a.X) + row * (int64_t)a.D, min(a.D, UN * TPR * 8), t, TPR);
    pdl_enter();
    if (row >= a.N) return;
    const int D = a.D;
    const int64_t off = row * (int64_t)D;
    if constexpr (VEC8) {
        // the first logits are requested before the per-row scalars are waited on
        float2 f[UN][4];
        ce_load<TPR, XT, UN>(a.X, off, t, D, f);
        const int64_t tg = a.T[row];
        const float g = ce_row_grad(a, row, tg);
        const float l = a.lse[row];
        const float scale = g * (1.f + 2.f * a.z * l);   // multiplies p = exp(x - lse)
        const float gq = g * a.eps / (float)D;            // g * (uniform part of q)
        const float gt = g * (1.f - a.eps);               // g * (target part of q)
        const int tc = (tg >= 0 && tg < D) ? (int)(tg >> 3) : -1;
        const float2 l2e = make_float2(kLog2e, kLog2e);
        const float2 nl2 = make_float2(-l * kLog2e, -l * kLog2e);
        const float2 scale2 = make_float2(scale, scale), ngq2 = make_float2(-gq, -gq);
        for (int c0 = t;;) {
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                const int c = c0 + u * TPR;
                if (c * 8 >= D) continue;
                float2 o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 e = __ffma2_rn(f[u][p], l2e, nl2);   // (x - lse) log2(e)
                    o[p] = __ffma2_rn(scale2, make_float2(ex2(e.x), ex2(e.y)), ngq2);
                }
                if (c == tc) {
                    const int e = (int)(tg & 7);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        o[p].x -= (e == 2 * p) ? gt : 0.f;
                        o[p].y -= (e == 2 * p + 1) ? gt : 0.f;
                    }
                }
                st_chunk<XT>(as<XT>(a.dX) + off + c * 8, o);
            }
            c0 += UN * TPR;
            if (c0 * 8 >= D) break;
            ce_load<TPR, XT, UN>(a.X, off, c0, D, f);
        }
    } else {
        const int64_t tg = a.T[row];
        const float g = ce_row_grad(a, row, tg);
        const float l = a.lse[row];
        const float scale = g * (1.f + 2.f * a.z * l);
        const float gq = g * a.eps / (float)D;
        const float gt = g * (1.f - a.eps);
        for (int j = t; j < D; j += TPR) {
            const float v = ld_elem_stream(a.X, off + j, a.xdt);
            st_elem(a.dX, off + j, scale * __expf(v - l) - gq - (j == tg ? gt : 0.f), a.xdt);
        }
    }
}

// ------------------------------------------------ softmax of wide rows (streaming) ---
// Rows wider than the register-resident softmax kernels hold (D > 16384; up to the
// 262144 columns of the meTile training_losses bounds): one CTA of TPR threads per row,
// two passes over the row, every combination in a fixed order.
//  * Forward: pass 1 keeps the running (maximum, sum of exp) state of the cross-entropy
//    forward (packed chunk maxima, one update per batch of UN chunks) and the CTA combines
//    it into lse = m + log(s); pass 2 reads the row again (mostly from L2: pass 1 reads
//    with the default cache policy) and writes y = exp(x - lse), or x - lse.
//  * Backward: pass 1 reduces sum dY*Y (softmax) or sum dY (log-softmax); pass 2 writes
//    dX = Y*(dY - sum) or dY - exp(Y)*sum.
//  * CLU (backward): a row is split over a thread-block cluster, CTA r taking columns
//    [r*slice, (r+1)*slice); the CTAs' sums are exchanged once through distributed
//    shared memory and added in rank order (cluster_sum), so every CTA gets the same
//    bits. Fewer rows are then in flight at once (the second read finds its slice in L2
//    more often), and a few hundred rows still make many CTAs. (The same split of the
//    forward measured slower on GB300: 256 x 262144 fp16 61.4 -> 68.8 - 92.8 us.)

// The 16-byte units of chunk c of the row at `off`, as loaded (zeros past the end).
template <int XT, int H>
__device__ __forceinline__ void ld_raw_chunk(const void *base, int64_t off, int c, int D,
                                             uint4 (&r)[chunk_units<XT>()]) {
    constexpr int CU = chunk_units<XT>();
#pragma unroll
    for (int q = 0; q < CU; ++q)
        r[q] = c * 8 < D ? ld_unit<H>(as<XT>(base) + off + c * 8 + q * (8 / CU)) : make_uint4(0, 0, 0, 0);
}

// Block-wide fixed-order combination of the (maximum, sum) states; every thread gets the
// total (every warp combines the same operands in the same lanes).
template <int TPR>
__device__ __forceinline__ MaxSum block_maxsum(MaxSum st, float *sm_m, float *sm_s) {
    constexpr int W = TPR / 32;
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum other{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.s, o)};
        st = (lane & o) ? combine(other, st) : combine(st, other);
    }
    if (lane == 0) {
        sm_m[w] = st.m;
        sm_s[w] = st.s;
    }
    __syncthreads();
    MaxSum tot{sm_m[lane & (W - 1)], sm_s[lane & (W - 1)]};  // W aligned groups, same operands
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
        MaxSum other{__shfl_xor_sync(0xffffffffu, tot.m, o), __shfl_xor_sync(0xffffffffu, tot.s, o)};
        tot = (lane & o) ? combine(other, tot) : combine(tot, other);
    }
    return tot;
}

// CIT > 0 (aligned rows): the first CIT batches of UN chunks a thread loads in the first
// pass are also kept in shared memory (CIT * UN * TPR 16-byte units per chunk unit, the
// dynamic shared memory of the launch), and the second pass takes them from there: only
// the rest of the row, the part read last, is read again from global memory, where it is
// the most likely to still be in L2. The shared memory also leaves one CTA per SM, so
// fewer rows are between their two passes at a time.
template <int TPR, bool VEC8, int XT, bool LOG, int UN, int MINB, int CIT = 0>
__global__ void __launch_bounds__(TPR, MINB)
softmax_stream_fwd_kernel(const SoftmaxArgs a) {
    constexpr int W = TPR / 32;
    static_assert(W <= 32 && (W & (W - 1)) == 0, "warps per row: a power of two up to 32");
    static_assert(CIT == 0 || VEC8, "the row cache holds aligned chunks");
    __shared__ float sm_m[W], sm_s[W];
    extern __shared__ __align__(16) uint4 xcache[];  // [CIT][UN][CU][TPR]
    const int t = threadIdx.x;
    const int64_t row = blockIdx.x;
    const int D = a.D;
    const int64_t off = row * (int64_t)D;
    if constexpr (VEC8) prefetch_l2(as<XT>(a.X) + off, min(D, UN * TPR * 8), t, TPR);  // (see ce_fwd_kernel)
    pdl_enter();
    constexpr int CU0 = VEC8 ? chunk_units<XT>() : 1;
    auto cache_at = [&](int it, int u, int q) -> uint4 & {
        return xcache[((it * UN + u) * CU0 + q) * TPR + t];
    };

    MaxSum st{-INFINITY, 0.f};
    if constexpr (VEC8) {
        constexpr int CU = chunk_units<XT>();
        const float2 l2e = make_float2(kLog2e, kLog2e);
        uint4 raw[UN][CU];
        ce_load_raw<TPR, XT, UN, kReadOnly>(a.X, off, t, D, raw);
        for (int c0 = t, it = 0;; ++it) {
            if (it < CIT) {
#pragma unroll
                for (int u = 0; u < UN; ++u)
#pragma unroll
                    for (int q = 0; q < CU; ++q) cache_at(it, u, q) = raw[u][q];
            }
            float bm = chunk_max<XT>(raw[0]);
#pragma unroll
            for (int u = 1; u < UN; ++u) bm = fmaxf(bm, chunk_max<XT>(raw[u]));
            const float m = fmaxf(st.m, bm);
            const float ms = (m == -INFINITY) ? 0.f : m;
            const float nb = -ms * kLog2e;
            const float2 nb2 = make_float2(nb, nb);
            st.s *= ex2(fmaf(st.m, kLog2e, nb));
            st.m = m;
            float2 cs2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                if ((c0 + u * TPR) * 8 >= D) continue;
                float2 f[4];
                unpack_chunk<XT, 4>(raw[u], 1, f);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 e = __ffma2_rn(f[p], l2e, nb2);
                    cs2 = __fadd2_rn(cs2, make_float2(ex2(e.x), ex2(e.y)));
                }
            }
            st.s += cs2.x + cs2.y;
            c0 += UN * TPR;
            if (c0 * 8 >= D) break;
            ce_load_raw<TPR, XT, UN, kReadOnly>(a.X, off, c0, D, raw);
        }
    } else {
        for (int j = t; j < D; j += TPR) add_value(st, ld_elem(a.X, off + j, a.xdt));
    }
    const MaxSum tot = block_maxsum<TPR>(st, sm_m, sm_s);
    const float lse = tot.m + logf(tot.s);

    if constexpr (VEC8) {
        const float2 l2e = make_float2(kLog2e, kLog2e);
        const float2 nl2 = make_float2(-lse * kLog2e, -lse * kLog2e);
        const float2 nlse = make_float2(-lse, -lse);
        constexpr int CU = chunk_units<XT>();
        for (int c0 = t, it = 0; c0 * 8 < D; c0 += UN * TPR, ++it) {
            uint4 raw[UN][CU];
            if (it < CIT) {
#pragma unroll
                for (int u = 0; u < UN; ++u)
#pragma unroll
                    for (int q = 0; q < CU; ++q) raw[u][q] = cache_at(it, u, q);
            } else {
                ce_load_raw<TPR, XT, UN>(a.X, off, c0, D, raw);
            }
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                const int c = c0 + u * TPR;
                if (c * 8 >= D) continue;
                float2 f[4];
                unpack_chunk<XT, 4>(raw[u], 1, f);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if constexpr (LOG) {
                        f[p] = __fadd2_rn(f[p], nlse);
                    } else {
                        const float2 e = __ffma2_rn(f[p], l2e, nl2);  // (x - lse) log2(e)
                        f[p] = make_float2(ex2(e.x), ex2(e.y));
                    }
                }
                st_chunk<XT>(as<XT>(a.Y) + off + c * 8, f);
            }
        }
    } else {
        for (int j = t; j < D; j += TPR) {
            const float v = ld_elem_stream(a.X, off + j, a.xdt);
            st_elem(a.Y, off + j, LOG ? v - lse : __expf(v - lse), a.xdt);
        }
    }
}

template <int TPR, bool VEC8, int XT, bool LOG, int UN, int MINB, bool CLU = false>
__global__ void __launch_bounds__(TPR, MINB)
softmax_stream_bwd_kernel(const SoftmaxArgs a) {
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * WPR];
    __shared__ float xch[1];  // cluster_sum's slot
    const int t = threadIdx.x, lane = t % 32, w = t / 32;
    // this CTA's columns: the row, or its slice of a split row, as a row of D columns
    const Window<CLU> win(a.D, a.slice);
    const int64_t row = win.owner();
    const int D = max(win.end - win.beg, 0);
    const int64_t off = row * (int64_t)a.D + win.beg;
    if constexpr (VEC8) {  // (see ce_fwd_kernel)
        prefetch_l2(as<XT>(a.X) + off, min(D, UN * TPR * 8), t, TPR);
        prefetch_l2(as<XT>(a.dY) + off, min(D, UN * TPR * 8), t, TPR);
    }
    pdl_enter();

    // pass 1: sum dY*Y (softmax) or sum dY (log-softmax). The chunks in flight stay as
    // loaded (16-byte units) until used: half the registers of fp32 pairs for 2-byte types.
    constexpr int CU = chunk_units<XT>();
    float v[1] = {0.f};
    if constexpr (VEC8) {
        float2 acc = make_float2(0.f, 0.f);
        for (int c0 = t; c0 * 8 < D; c0 += UN * TPR) {
            uint4 yr[LOG ? 1 : UN][CU], gr[UN][CU];
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                ld_raw_chunk<XT, kReadOnly>(a.dY, off, c0 + u * TPR, D, gr[u]);
                if constexpr (!LOG) ld_raw_chunk<XT, kReadOnly>(a.X, off, c0 + u * TPR, D, yr[u]);
            }
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                float2 gv[4], yv[4];
                unpack_chunk<XT, 4>(gr[u], 1, gv);
                if constexpr (!LOG) unpack_chunk<XT, 4>(yr[u], 1, yv);
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    acc = LOG ? __fadd2_rn(acc, gv[p]) : __ffma2_rn(gv[p], yv[p], acc);
            }
        }
        v[0] = acc.x + acc.y;
    } else {
        for (int j = t; j < D; j += TPR) {
            const float g = ld_elem(a.dY, off + j, a.gdt);
            v[0] += LOG ? g : g * ld_elem(a.X, off + j, a.xdt);
        }
    }
    row_sum<TPR, 1, 1>(v, red, 0, 0, w, lane);
    if constexpr (CLU) {
        cluster_sum<1>(v, xch, 0, win.cn);
        cluster_arrive();  // done reading the other CTAs' slots (waited for before exit)
    }
    const float c = v[0];

    // pass 2: dX
    if constexpr (VEC8) {
        const float2 nc = make_float2(-c, -c);
        for (int c0 = t; c0 * 8 < D; c0 += UN * TPR) {
            uint4 yr[UN][CU], gr[UN][CU];
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                ld_raw_chunk<XT, kStream>(a.X, off, c0 + u * TPR, D, yr[u]);
                ld_raw_chunk<XT, kStream>(a.dY, off, c0 + u * TPR, D, gr[u]);
            }
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                const int ch = c0 + u * TPR;
                if (ch * 8 >= D) continue;
                float2 yk[4], gk[4];
                unpack_chunk<XT, 4>(yr[u], 1, yk);
                unpack_chunk<XT, 4>(gr[u], 1, gk);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if constexpr (LOG) {
                        const float2 e = make_float2(__expf(yk[p].x), __expf(yk[p].y));
                        gk[p] = __ffma2_rn(e, nc, gk[p]);                 // dY - exp(Y) c
                    } else {
                        gk[p] = __fmul2_rn(yk[p], __fadd2_rn(gk[p], nc));  // Y (dY - c)
                    }
                }
                st_chunk<XT>(as<XT>(a.Y) + off + ch * 8, gk);
            }
        }
    } else {
        for (int j = t; j < D; j += TPR) {
            const float y = ld_elem_stream(a.X, off + j, a.xdt);
            const float g = ld_elem_stream(a.dY, off + j, a.gdt);
            st_elem(a.Y, off + j, LOG ? g - __expf(y) * c : y * (g - c), a.xdt);
        }
    }
    if constexpr (CLU) cluster_wait();  // no CTA leaves while another may read its slots
}

// Fixed-order reduction of the per-row losses for sum/mean: one block; thread i sums rows
// i, i + B, ... in order (four rows' loads in flight) and counts the rows whose target is
// not ignore_index; then each warp's threads by a butterfly, and the warps' totals by a
// butterfly in warp 0 (the same order every run). The count is an integer (exact for any
// N < 2^32). out[0] = sum (reduction 1) or sum / count (2, divided in fp64 and rounded
// once; 0 when no row is valid), n_valid[0] = count rounded to fp32 (exact up to 2^24).
template <int B>
__global__ void __launch_bounds__(B)
ce_loss_reduce_kernel(const float *loss, const int64_t *T, int64_t N, int64_t ignore_index,
                      int reduction, float *out, float *n_valid) {
    pdl_enter();
    constexpr int W = B / 32, U = 4;
    static_assert(W <= 32 && W * 32 == B, "one warp adds the warp totals");
    __shared__ float ws[W];
    __shared__ unsigned wc[W];
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
    // per thread: rows threadIdx.x, + B, + 2B, ... in that order, U rows' loads in flight
    float s = 0.f;
    unsigned c = 0u;
    for (int64_t i0 = threadIdx.x; i0 < N; i0 += (int64_t)U * B) {
        float l[U];
        unsigned v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * B;
            l[u] = i < N ? loss[i] : 0.f;
            v[u] = (i < N && T[i] != ignore_index) ? 1u : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + (int64_t)u * B < N) {
                s += l[u];
                c += v[u];
            }
    }
    // the warp's threads by a butterfly, then the warp totals in warp order
    s = warp_sum(s);
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) {
        ws[w] = s;
        wc[w] = c;
    }
    __syncthreads();
    if (w == 0) {
        const float tot = warp_sum(lane < W ? ws[lane] : 0.f);
        const unsigned cnt = __reduce_add_sync(0xffffffffu, lane < W ? wc[lane] : 0u);
        if (lane == 0) {
            out[0] = (reduction == 2) ? (cnt > 0u ? (float)((double)tot / (double)cnt) : 0.f) : tot;
            n_valid[0] = (float)cnt;
        }
    }
}

}  // namespace mt
