// gemv.cuh -- fused normalization + GEMV for decode (tensorcore "Training kernels", "Fused
// Norm + GEMV"): Y[M, N] = Norm(X[M, K], gamma[, beta]) @ W[K, N], with Norm the RMSNorm or
// LayerNorm forward, fp16 storage, fp32 arithmetic, the normalized rows applied in
// registers and never stored. M is small (decode batches; up to 8 here).
//
// The work is HBM-bound on W: each 2-byte weight feeds M multiply-adds, at most 8 flops per
// byte for M = 8, two orders of magnitude under the tensor-core ridge. So W is streamed
// once with 16-byte loads and the products are fp32x2 FMAs on the CUDA cores. Two
// launches, chained by programmatic dependent launch:
//
//  1. gemv_stats_kernel: the M rows' statistics (RMSNorm: mean of squares; LayerNorm:
//     mean, then the centred second moment, two passes from registers), one CTA per row,
//     as the page's pass 1 (rstd computed inline, no normalized row written back).
//  2. norm_gemv_kernel: split-K partial products. The output columns are cut into tiles
//     of TILE = 8 * LPF and the input features into KS slices; CTA (tile, slice) streams
//     the slice's rows of its tile of W. LPF lanes cover a tile (lane l: columns 8l ..
//     8l+7, one 16-byte chunk of a W row; LPF = 32: 512 contiguous bytes per warp load)
//     and a warp takes G = 32 / LPF features per step. Each thread copies its own W
//     chunks with cp.async into a shared-memory ring S - 1 features ahead and reads back
//     only what it copied (cp.async.wait_group alone orders the ring). The copies start
//     before the kernel waits for the statistics: W is not written by the kernels before
//     it. The slice of the normalized rows is built in shared memory, fp32 (the page's
//     pass 2: normalization applied during the accumulation).
//     The last CTA to finish a column tile (counted with one atomic increment per CTA on
//     the tile's counter, after a fence that publishes its partial sums) adds the KS
//     partial rows of the tile in slice order and writes Y, rounded to fp16 (the loads of
//     a batch of slices for all of a thread's outputs are issued before their adds). Nothing
//     waits on the counter: the other CTAs just exit.
//
// Deterministic sums: per thread, features in ascending order; the G feature groups of a
// warp by a butterfly; the warps of a CTA in warp order; the slices in slice order (the
// counter only elects which CTA adds them). Y is bitwise reproducible.
#pragma once

#include "pipe.cuh"

namespace mt {

struct GemvArgs {
    const void *X;      // [M, K] fp16
    const void *gamma;  // [K] fp16
    const void *beta;   // [K] fp16 (LayerNorm only)
    const void *W;      // [K, N] fp16, row k = the weights of input feature k
    void *Y;            // [M, N] fp16
    float *stats;       // [M][2]: mean (0 for RMSNorm), rstd
    float *part;        // [KS][M][N] fp32 partial products
    unsigned *count;    // [tiles] finished slices per column tile (zeroed by the stats kernel)
    int tiles;          // column tiles
    int M, N, K;
    int slice;          // input features per slice (a multiple of 8)
    int ks;             // slices
    float eps;
    int xvec;           // X, gamma, beta take 16-byte loads (K % 8 == 0, aligned bases)
};

constexpr int kGemvMaxRows = 8;
constexpr int kGemvWarps = 8;
constexpr int kGemvStatsThreads = 1024;
// 8-element chunks of a row per stats thread (K <= 8 * 1024 * 4 = 32768) and of a slice
// per GEMV thread (slice <= 8 * 256 * 2 = 4096).
constexpr int kGemvRowChunks = 4;
constexpr int kGemvSliceChunks = 2;

// Rows padded to the shared-memory stride of the normalized features (float4 loads).
template <int MT>
__host__ __device__ constexpr int gemv_mp() { return MT <= 4 ? 4 : 8; }

// Shared memory of a GEMV launch: the normalized slice, then the W ring (S stages of one
// 16-byte chunk per thread), reused after the stream for the warps' partial sums.
#ifndef MT_GEMV_CPL
#define MT_GEMV_CPL 1
#endif
// 16-byte chunks per lane and feature: lane l's chunks sit 8 * LPF columns apart, so each
// warp load instruction still covers 16 * LPF contiguous bytes.
constexpr int kGemvCpl = MT_GEMV_CPL;

template <int MT, int LPF, int S>
constexpr size_t gemv_smem(int slice) {
    const size_t ring = (size_t)S * kGemvCpl * kGemvWarps * 32 * 16;
    const size_t red = (size_t)kGemvWarps * MT * (8 * LPF * kGemvCpl) * sizeof(float);
    return (size_t)slice * gemv_mp<MT>() * sizeof(float) + (ring > red ? ring : red);
}

// Eight consecutive fp16 values p[k0 .. k0+7] (zeros past `end`): one 16-byte load when
// VEC (k0 a multiple of 8, p 16-byte aligned), else per-element loads.
template <bool VEC>
__device__ __forceinline__ uint4 gemv_ld8(const __half *p, int k0, int end) {
    if (k0 >= end) return make_uint4(0, 0, 0, 0);
    if constexpr (VEC) {
        return ld_unit<kReadOnly>(p + k0);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const unsigned short lo = k0 + 2 * i < end ? __half_as_ushort(p[k0 + 2 * i]) : 0;
            const unsigned short hi = k0 + 2 * i + 1 < end ? __half_as_ushort(p[k0 + 2 * i + 1]) : 0;
            w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One 16-byte chunk (8 fp16 columns) of W row k at column col; VEC: aligned 16-byte load,
// otherwise per-element loads with the columns past N reading 0.
template <bool VEC>
__device__ __forceinline__ uint4 gemv_ld_w(const __half *W, int64_t k, int N, int col) {
    const __half *p = W + k * (int64_t)N + col;
    if constexpr (VEC) {
        return ld_unit<kStream>(p);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const unsigned short lo = col + 2 * i < N ? __half_as_ushort(p[2 * i]) : 0;
            const unsigned short hi = col + 2 * i + 1 < N ? __half_as_ushort(p[2 * i + 1]) : 0;
            w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 1. Row statistics: CTA m (kGemvStatsThreads threads) reduces row m of X.
template <int OP>
__global__ void __launch_bounds__(kGemvStatsThreads)
gemv_stats_kernel(const GemvArgs a) {
    constexpr int T = kGemvStatsThreads;
    __shared__ float red[2 * (T / 32)];
    pdl_enter();
    const int tid = threadIdx.x, m = blockIdx.x, K = a.K;
    const __half *x = static_cast<const __half *>(a.X) + (int64_t)m * K;
    uint4 raw[kGemvRowChunks];
#pragma unroll
    for (int c = 0; c < kGemvRowChunks; ++c) {
        const int k0 = 8 * (tid + c * T);
        raw[c] = a.xvec ? gemv_ld8<true>(x, k0, K) : gemv_ld8<false>(x, k0, K);
    }
    float v[1] = {0.f};
#pragma unroll
    for (int c = 0; c < kGemvRowChunks; ++c) {
        float2 f[4];
        unpack_unit<kF16>(raw[c], f);
#pragma unroll
        for (int p = 0; p < 4; ++p) v[0] += (OP == kLayer) ? f[p].x + f[p].y : f[p].x * f[p].x + f[p].y * f[p].y;
    }
    row_sum<T, 1, 1>(v, red, 0, 0, tid / 32, tid % 32);
    float mu = 0.f;
    if constexpr (OP == kLayer) {
        mu = v[0] / (float)K;
        v[0] = 0.f;
#pragma unroll
        for (int c = 0; c < kGemvRowChunks; ++c) {
            const int k0 = 8 * (tid + c * T);
            float2 f[4];
            unpack_unit<kF16>(raw[c], f);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float dx = k0 + 2 * p < K ? f[p].x - mu : 0.f;
                const float dy = k0 + 2 * p + 1 < K ? f[p].y - mu : 0.f;
                v[0] += dx * dx + dy * dy;
            }
        }
        row_sum<T, 1, 1>(v, red, 1, 0, tid / 32, tid % 32);
    }
    if (tid == 0) {
        a.stats[2 * m] = mu;
        a.stats[2 * m + 1] = rsqrtf(v[0] / (float)K + a.eps);
    }
    if (m == 0)
        for (int t = tid; t < a.tiles; t += T) a.count[t] = 0u;
}

// 2. Split-K partial products. OP: kRms or kLayer. MT: rows the kernel is compiled for
// (M <= MT; rows past M are zero and not stored). LPF: lanes per feature (32, 16 or 8).
// S: W ring stages (VEC only). grid = ceil(N / TILE) * KS CTAs of kGemvWarps warps.
template <int OP, int MT, int LPF, int S, bool VEC>
__global__ void __launch_bounds__(kGemvWarps * 32, 2)
norm_gemv_kernel(const GemvArgs a) {
    constexpr int THREADS = kGemvWarps * 32;
    constexpr int G = 32 / LPF;              // features per warp step
    constexpr int FG = kGemvWarps * G;       // feature groups per CTA
    constexpr int CPL = kGemvCpl;            // chunks per lane and feature
    constexpr int TILE = 8 * LPF * CPL;      // output columns per CTA
    constexpr int MP = gemv_mp<MT>();
    static_assert(OP == kRms || OP == kLayer, "RMSNorm or LayerNorm");
    static_assert(MT >= 1 && MT <= kGemvMaxRows && (LPF == 32 || LPF == 16 || LPF == 8), "shape");
    extern __shared__ __align__(16) float gsm[];

    const int tid = threadIdx.x, w = tid / 32, lane = tid % 32;
    const int M = a.M, N = a.N, K = a.K;
    // CTA b: tile b % tiles of slice b / tiles (neighbouring CTAs read neighbouring
    // stretches of the same W rows)
    const int ntiles = (N + TILE - 1) / TILE;
    const int tile = (int)(blockIdx.x % ntiles), ks = (int)(blockIdx.x / ntiles);
    const int kbeg = ks * a.slice, kend = min(K, kbeg + a.slice);
    const int f = w * G + lane / LPF;                 // this thread's feature group
    const int col = tile * TILE + (lane % LPF) * 8;   // first column of its chunk 0
    const int nk = kbeg + f < kend ? (kend - kbeg - f + FG - 1) / FG : 0;  // its features
    const __half *W = static_cast<const __half *>(a.W);
    float *xn = gsm;                                                      // [slice][MP]
    uint4 *ring = reinterpret_cast<uint4 *>(gsm + (size_t)a.slice * MP);  // [S][THREADS]

    // start the W stream (before the wait: no earlier kernel of the chain writes W)
    auto issue = [&](int i) {
        if constexpr (VEC) {
            if (i < nk) {
#pragma unroll
                for (int c = 0; c < CPL; ++c)
                    if (col + c * 8 * LPF < N)
                        cp_async16(smem_addr(&ring[((i % S) * CPL + c) * THREADS + tid]),
                                   W + (int64_t)(kbeg + f + i * FG) * N + col + c * 8 * LPF);
            }
            cp_async_commit();
        }
    };
#pragma unroll
    for (int i = 0; i < S - 1; ++i) issue(i);
    // RMSNorm factors rstd out of the sums: Y = rstd * sum_k (x_k g_k) W_k, so the slice
    // x * g needs no statistics and the kernel waits for the statistics kernel only before
    // it counts its tile (the wait also covers the tile counters that kernel zeroes). X is
    // visible already: this kernel launches only once the statistics kernel has passed its
    // own wait for the kernel that wrote X. LayerNorm builds the normalized slice, so it
    // waits here.
    if constexpr (OP == kRms) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    else pdl_enter();  // the statistics are complete and visible from here on

    // the slice: thread t builds features of chunks t and t + THREADS
    const __half *X = static_cast<const __half *>(a.X);
    const __half *gam = static_cast<const __half *>(a.gamma);
    const __half *bet = static_cast<const __half *>(a.beta);
    float mu[MT], rs[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        mu[m] = (OP == kLayer && m < M) ? a.stats[2 * m] : 0.f;
        rs[m] = (OP == kLayer && m < M) ? a.stats[2 * m + 1] : 1.f;
    }
#pragma unroll
    for (int c = 0; c < kGemvSliceChunks; ++c) {
        const int k0 = kbeg + 8 * (tid + c * THREADS);
        if (k0 >= kend) continue;
        float2 g2[4], b2[4], x2[MT][4];
        unpack_unit<kF16>(a.xvec ? gemv_ld8<true>(gam, k0, kend) : gemv_ld8<false>(gam, k0, kend), g2);
        if constexpr (OP == kLayer)
            unpack_unit<kF16>(a.xvec ? gemv_ld8<true>(bet, k0, kend) : gemv_ld8<false>(bet, k0, kend), b2);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint4 r = m < M ? (a.xvec ? gemv_ld8<true>(X + (int64_t)m * K, k0, kend)
                                            : gemv_ld8<false>(X + (int64_t)m * K, k0, kend))
                                  : make_uint4(0, 0, 0, 0);
            unpack_unit<kF16>(r, x2[m]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int k = k0 + e;
            if (k >= kend) break;
            const float g = (e & 1) ? g2[e / 2].y : g2[e / 2].x;
            const float b = (OP == kLayer) ? ((e & 1) ? b2[e / 2].y : b2[e / 2].x) : 0.f;
            float v[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                v[m] = 0.f;
                if (m < MT && m < M) {
                    const float xv = (e & 1) ? x2[m][e / 2].y : x2[m][e / 2].x;
                    v[m] = (xv - mu[m]) * rs[m] * g + b;
                }
            }
#pragma unroll
            for (int qd = 0; qd < MP / 4; ++qd)
                reinterpret_cast<float4 *>(xn + (size_t)(k - kbeg) * MP)[qd] =
                    make_float4(v[4 * qd], v[4 * qd + 1], v[4 * qd + 2], v[4 * qd + 3]);
        }
    }
    __syncthreads();

    // stream: acc[m][p] += xn[k][m] * W[k][col + 2p .. 2p+1], features ascending
    float2 acc[CPL][MT][4];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[c][m][p] = make_float2(0.f, 0.f);
    for (int i = 0; i < nk; ++i) {
        uint4 raw[CPL];
        if constexpr (VEC) {
            issue(i + S - 1);
            cp_async_wait<S - 1>();  // this thread's copies of feature i have landed
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                raw[c] = col + c * 8 * LPF < N ? ring[((i % S) * CPL + c) * THREADS + tid]
                                               : make_uint4(0, 0, 0, 0);
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                raw[c] = col + c * 8 * LPF < N
                             ? gemv_ld_w<false>(W, kbeg + f + (int64_t)i * FG, N, col + c * 8 * LPF)
                             : make_uint4(0, 0, 0, 0);
        }
        const int kl = f + i * FG;  // feature index within the slice
        float xv[MP];
#pragma unroll
        for (int q = 0; q < MP / 4; ++q) {
            const float4 t = reinterpret_cast<const float4 *>(xn + (size_t)kl * MP)[q];
            xv[4 * q] = t.x;
            xv[4 * q + 1] = t.y;
            xv[4 * q + 2] = t.z;
            xv[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            float2 wf[4];
            unpack_unit<kF16>(raw[c], wf);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float2 x2 = make_float2(xv[m], xv[m]);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[c][m][p] = __ffma2_rn(x2, wf[p], acc[c][m][p]);
            }
        }
    }
    if constexpr (VEC) cp_async_wait<0>();

    // fixed-order sums: the warp's feature groups (butterfly over lane / LPF), then the
    // CTA's warps (shared memory, warp order); one partial row per (slice, row m)
#pragma unroll
    for (int o = LPF; o < 32; o <<= 1)
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    acc[c][m][p].x += __shfl_xor_sync(0xffffffffu, acc[c][m][p].x, o);
                    acc[c][m][p].y += __shfl_xor_sync(0xffffffffu, acc[c][m][p].y, o);
                }
    __syncthreads();  // every thread is done with its ring slots
    float *wpart = reinterpret_cast<float *>(ring);  // [kGemvWarps][MT][TILE]
    if (lane < LPF) {
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float4 *dst = reinterpret_cast<float4 *>(wpart + ((size_t)w * MT + m) * TILE +
                                                         lane * 8 + c * 8 * LPF);
                dst[0] = make_float4(acc[c][m][0].x, acc[c][m][0].y, acc[c][m][1].x, acc[c][m][1].y);
                dst[1] = make_float4(acc[c][m][2].x, acc[c][m][2].y, acc[c][m][3].x, acc[c][m][3].y);
            }
    }
    __syncthreads();
    for (int idx = tid; idx < M * TILE; idx += THREADS) {
        const int m = idx / TILE, c = idx % TILE, n = tile * TILE + c;
        if (n >= N) continue;
        float sum = wpart[(size_t)m * TILE + c];
#pragma unroll
        for (int ww = 1; ww < kGemvWarps; ++ww) sum += wpart[((size_t)ww * MT + m) * TILE + c];
        a.part[((size_t)ks * M + m) * N + n] = sum;
    }

    // the last of the tile's KS CTAs adds the partial rows in slice order
    __shared__ unsigned last;
    if constexpr (OP == kRms) asm volatile("griddepcontrol.wait;" ::: "memory");
    __threadfence();  // publish this CTA's partial rows before counting it
    __syncthreads();
    if (tid == 0) last = (atomicAdd(&a.count[tile], 1u) == (unsigned)a.ks - 1u);
    __syncthreads();
    if (!last) return;
    __threadfence();
    // Each thread owns outputs idx = tid + i * THREADS (i < OUTS) and adds each one's KS
    // partials in slice order; the loads of SB slices of all its outputs are issued before
    // their adds, so that they are in flight together (the same sums as one add at a time).
    constexpr int OUTS = (MT * TILE + THREADS - 1) / THREADS;
    constexpr int SB = (32 / OUTS) > 0 ? 32 / OUTS : 1;
    __half *Y = static_cast<__half *>(a.Y);
    const size_t step = (size_t)M * N;
    float sum[OUTS];
    const float *src[OUTS];
    bool on[OUTS];
#pragma unroll
    for (int i = 0; i < OUTS; ++i) {
        const int idx = tid + i * THREADS;
        const int m = idx / TILE, n = tile * TILE + idx % TILE;
        on[i] = idx < M * TILE && n < N;
        src[i] = a.part + (size_t)(on[i] ? m : 0) * N + (on[i] ? n : 0);
        sum[i] = 0.f;
    }
    for (int k0 = 0; k0 < a.ks; k0 += SB) {
        float v[OUTS][SB];
#pragma unroll
        for (int i = 0; i < OUTS; ++i)
#pragma unroll
            for (int b = 0; b < SB; ++b)
                v[i][b] = (on[i] && k0 + b < a.ks) ? __ldcg(src[i] + (size_t)(k0 + b) * step) : 0.f;
#pragma unroll
        for (int i = 0; i < OUTS; ++i)
#pragma unroll
            for (int b = 0; b < SB; ++b)
                if (k0 + b < a.ks) sum[i] += v[i][b];
    }
#pragma unroll
    for (int i = 0; i < OUTS; ++i) {
        const int idx = tid + i * THREADS;
        if (on[i]) {
            const int m = idx / TILE;
            const float r = (OP == kRms) ? a.stats[2 * m + 1] : 1.f;  // RMSNorm: rstd applied here
            Y[(int64_t)m * N + tile * TILE + idx % TILE] = __float2half_rn(sum[i] * r);
        }
    }
}

}  // namespace mt
