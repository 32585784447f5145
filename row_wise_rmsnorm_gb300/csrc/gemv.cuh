// gemv.cuh -- fused normalization + GEMV for decode (tensorcore "Training kernels", "Fused
// Norm + GEMV"): Y[M, N] = Norm(X[M, K], gamma[, beta]) @ W[K, N], with Norm the RMSNorm or
// LayerNorm forward, fp16 storage, fp32 arithmetic, the normalized rows applied in
// registers and never stored. M is small (decode batches; up to 8 here).
//
// The work is HBM-bound on W: each 2-byte weight feeds M multiply-adds, at most 8 flops per
// byte for M = 8, two orders of magnitude under the tensor-core ridge. So W is streamed
// once with 16-byte loads and the products are fp32x2 FMAs on the CUDA cores.
//
//  * Tiles. A CTA owns a tile of TILE = 8 * LPF output columns and a slice of the K input
//    features. LPF lanes cover the tile (lane l: columns 8l .. 8l+7, one 16-byte chunk of a
//    W row); a warp takes G = 32 / LPF features per step (LPF = 32: 512 contiguous bytes of
//    one W row per warp load; LPF = 16: 256 bytes of each of two rows), and the CTA's
//    feature groups take features beg + f, beg + f + FG, ... of its slice.
//  * Clusters along K. The CL CTAs of a column tile form a thread-block cluster; rank r
//    takes features [r * slice, (r + 1) * slice).
//  * Statistics inline. Each CTA loads its slice of the M rows of X (one batch of 16-byte
//    loads per thread), sums it, and the cluster's CTAs combine the row statistics in one
//    exchange through distributed shared memory, as a split normalization row does
//    (RMSNorm: sums of squares; LayerNorm: slice sums and centred second moments
//    combined by the within/between-slice identity). Each thread then writes its
//    features of the normalized rows, fp32, to shared memory (the page's "compute rstd
//    inline ... skip the write-back").
//  * W through a per-thread ring. Each thread copies its own 16-byte W chunks with
//    cp.async into a shared-memory ring S - 1 features ahead and reads back only what it
//    copied, so cp.async.wait_group alone orders the ring (no barrier, no mbarrier) and
//    the bytes in flight are set by the ring depth, not by registers. The stream starts
//    before the statistics are computed. (Rows not 16-byte aligned, or N % 8 != 0, load
//    per element without the ring.)
//  * Deterministic sums. Per thread, features in ascending order; then the G feature
//    groups of a warp by a butterfly, the warps of a CTA in warp order (shared memory),
//    the CTAs of a cluster in rank order (distributed shared memory). No atomics: every
//    output is bitwise reproducible.
#pragma once

#include "pipe.cuh"

namespace mt {

struct GemvArgs {
    const void *X;      // [M, K] fp16
    const void *gamma;  // [K] fp16
    const void *beta;   // [K] fp16 (LayerNorm only)
    const void *W;      // [K, N] fp16, row k = the weights of input feature k
    void *Y;            // [M, N] fp16
    int M, N, K;
    int slice;          // features per CTA of a cluster (a multiple of 8)
    float eps;
    int xvec;           // X, gamma, beta take 16-byte loads (K % 8 == 0, aligned bases)
};

constexpr int kGemvMaxRows = 8;
constexpr int kGemvWarps = 8;
// 8-feature chunks of a CTA's slice per thread (a slice holds at most 8 * 256 * 2 = 4096
// features).
constexpr int kGemvSliceChunks = 2;

// LayerNorm statistics of MT split rows in one cluster exchange (the multi-row form of
// cluster_ln_stats): s[m] (slice sum) and q[m] (slice centred second moment) in, the row
// means and centred sums of squares out. xch: 4 * MT shared floats.
template <int MT>
__device__ __forceinline__ void cluster_ln_stats_rows(float (&s)[MT], float (&q)[MT], float *xch,
                                                      unsigned n, int K, int slice) {
    if (threadIdx.x == 0) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            xch[2 * m] = s[m];
            xch[2 * m + 1] = q[m];
        }
    }
    cluster_arrive();
    cluster_wait();
    const unsigned lane = threadIdx.x & 31u;
    float nr = 0.f;
    if (lane < n) {
        const int beg = (int)lane * slice;
        nr = (float)max(0, min(K, beg + slice) - beg);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float sr = lane < n ? ld_cluster(xch + 2 * m, lane) : 0.f;
        const float qr = lane < n ? ld_cluster(xch + 2 * m + 1, lane) : 0.f;
        const float mu = warp_sum(sr) / (float)K;
        const float dev = nr > 0.f ? sr / nr - mu : 0.f;
        s[m] = mu;
        q[m] = warp_sum(qr + nr * dev * dev);
    }
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

// Rows padded to the shared-memory stride of the normalized features (float4 loads).
template <int MT>
__host__ __device__ constexpr int gemv_mp() { return MT <= 4 ? 4 : 8; }

// Shared memory of a launch: the normalized slice and the W ring (S stages of one 16-byte
// chunk per thread), later reused for the warps' partials.
template <int MT, int LPF, int S>
constexpr size_t gemv_smem(int slice) {
    const size_t xn = (size_t)slice * gemv_mp<MT>() * sizeof(float);
    const size_t ring = (size_t)S * kGemvWarps * 32 * 16;
    const size_t red = (size_t)kGemvWarps * MT * (8 * LPF) * sizeof(float);
    return xn + ring > red ? xn + ring : red;
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

// OP: kRms or kLayer. MT: rows the kernel is compiled for (M <= MT; rows past M are zero
// and not stored). LPF: lanes per feature (32, 16 or 8). S: W ring stages (VEC only).
// grid = ceil(N / TILE) * CL CTAs of kGemvWarps warps, clusters of CL along x.
template <int OP, int MT, int LPF, int S, bool VEC>
__global__ void __launch_bounds__(kGemvWarps * 32, MT <= 4 ? 2 : 1)
norm_gemv_kernel(const GemvArgs a) {
    constexpr int THREADS = kGemvWarps * 32;
    constexpr int G = 32 / LPF;              // features per warp step
    constexpr int FG = kGemvWarps * G;       // feature groups per CTA
    constexpr int TILE = 8 * LPF;            // output columns per CTA
    constexpr int MP = gemv_mp<MT>();
    static_assert(OP == kRms || OP == kLayer, "RMSNorm or LayerNorm");
    static_assert(MT >= 1 && MT <= kGemvMaxRows && (LPF == 32 || LPF == 16 || LPF == 8), "shape");
    extern __shared__ __align__(16) float gsm[];
    __shared__ float red[2 * kGemvWarps * MT];
    __shared__ float xch[4 * MT];
    pdl_enter();

    const int tid = threadIdx.x, w = tid / 32, lane = tid % 32;
    const int M = a.M, N = a.N, K = a.K;
    const unsigned cn = cluster_size(), rank = cluster_rank();
    const int tile = (int)(blockIdx.x / cn);
    const int kbeg = (int)rank * a.slice, kend = min(K, kbeg + a.slice);
    const int f = w * G + lane / LPF;                 // this thread's feature group
    const int col = tile * TILE + (lane % LPF) * 8;   // first of its 8 columns
    const bool cok = col < N;
    const int nk = kbeg + f < kend ? (kend - kbeg - f + FG - 1) / FG : 0;  // its features
    const __half *W = static_cast<const __half *>(a.W);

    // 1. start the W stream: features i = 0 .. S-2 of this thread into ring slots i % S
    float *xn = gsm;                                           // [slice][MP]
    uint4 *ring = reinterpret_cast<uint4 *>(gsm + (size_t)a.slice * MP);  // [S][THREADS]
    auto issue = [&](int i) {
        if constexpr (VEC) {
            if (i < nk && cok)
                cp_async16(smem_addr(&ring[(i % S) * THREADS + tid]),
                           W + (int64_t)(kbeg + f + i * FG) * N + col);
            cp_async_commit();
        }
    };
#pragma unroll
    for (int i = 0; i < S - 1; ++i) issue(i);

    // 2. this CTA's slice of the rows of X (thread t: chunks t and t + 256 of the slice),
    //    row statistics (CTA sums, then one cluster exchange), the normalized slice
    const __half *X = static_cast<const __half *>(a.X);
    const __half *gam = static_cast<const __half *>(a.gamma);
    const __half *bet = static_cast<const __half *>(a.beta);
    uint4 xr[MT][kGemvSliceChunks];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int c = 0; c < kGemvSliceChunks; ++c) {
            const int k0 = kbeg + 8 * (tid + c * THREADS);
            xr[m][c] = make_uint4(0, 0, 0, 0);
            if (m < M)
                xr[m][c] = a.xvec ? gemv_ld8<true>(X + (int64_t)m * K, k0, kend)
                                  : gemv_ld8<false>(X + (int64_t)m * K, k0, kend);
        }
    float mu[MT], rs[MT];
    {
        float s[MT], q[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            s[m] = 0.f;
#pragma unroll
            for (int c = 0; c < kGemvSliceChunks; ++c) {
                float2 f2[4];
                unpack_unit<kF16>(xr[m][c], f2);
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    s[m] += (OP == kLayer) ? f2[p].x + f2[p].y : f2[p].x * f2[p].x + f2[p].y * f2[p].y;
            }
        }
        row_sum<THREADS, 1, MT>(s, red, 0, 0, w, lane);
        if constexpr (OP == kLayer) {
            // centre on the slice mean, from registers (zero-filled features are skipped)
            const float inv_n = 1.f / (float)max(kend - kbeg, 1);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float lm = s[m] * inv_n;
                q[m] = 0.f;
#pragma unroll
                for (int c = 0; c < kGemvSliceChunks; ++c) {
                    const int k0 = kbeg + 8 * (tid + c * THREADS);
                    float2 f2[4];
                    unpack_unit<kF16>(xr[m][c], f2);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const float dx = k0 + 2 * p < kend ? f2[p].x - lm : 0.f;
                        const float dy = k0 + 2 * p + 1 < kend ? f2[p].y - lm : 0.f;
                        q[m] += dx * dx + dy * dy;
                    }
                }
            }
            row_sum<THREADS, 1, MT>(q, red, 1, 0, w, lane);
            if (cn > 1) {
                cluster_ln_stats_rows<MT>(s, q, xch, cn, K, a.slice);  // s: means, q: M2
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) s[m] *= inv_n;
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                mu[m] = s[m];
                rs[m] = rsqrtf(q[m] / (float)K + a.eps);
            }
        } else {
            if (cn > 1) cluster_sum<MT>(s, xch, 0, cn);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                mu[m] = 0.f;
                rs[m] = rsqrtf(s[m] / (float)K + a.eps);
            }
        }
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
        for (int m = 0; m < MT; ++m) unpack_unit<kF16>(xr[m][c], x2[m]);
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

    // 3. stream W: acc[m][p] += xn[k][m] * W[k][col + 2p .. 2p+1], features ascending
    float2 acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[m][p] = make_float2(0.f, 0.f);
    for (int i = 0; i < nk; ++i) {
        uint4 raw;
        if constexpr (VEC) {
            issue(i + S - 1);
            cp_async_wait<S - 1>();  // this thread's copy of feature i has landed
            raw = ring[(i % S) * THREADS + tid];
        } else {
            raw = cok ? gemv_ld_w<false>(W, kbeg + f + (int64_t)i * FG, N, col) : make_uint4(0, 0, 0, 0);
        }
        const int kl = f + i * FG;  // feature index within the slice
        float2 wf[4];
        unpack_unit<kF16>(raw, wf);
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
        for (int m = 0; m < MT; ++m) {
            const float2 x2 = make_float2(xv[m], xv[m]);
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[m][p] = __ffma2_rn(x2, wf[p], acc[m][p]);
        }
    }
    if constexpr (VEC) cp_async_wait<0>();

    // 4. fixed-order sums: the warp's feature groups (butterfly over lane / LPF), then
    //    the CTA's warps (shared memory, warp order), then the cluster (rank order)
#pragma unroll
    for (int o = LPF; o < 32; o <<= 1)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                acc[m][p].x += __shfl_xor_sync(0xffffffffu, acc[m][p].x, o);
                acc[m][p].y += __shfl_xor_sync(0xffffffffu, acc[m][p].y, o);
            }
    __syncthreads();  // every warp is done with xn
    float *part = gsm;  // [kGemvWarps][MT][TILE]
    if (lane < LPF) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float4 *dst = reinterpret_cast<float4 *>(part + ((size_t)w * MT + m) * TILE + lane * 8);
            dst[0] = make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
            dst[1] = make_float4(acc[m][2].x, acc[m][2].y, acc[m][3].x, acc[m][3].y);
        }
    }
    __syncthreads();
    for (int c = tid; c < TILE; c += THREADS) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float s = part[(size_t)m * TILE + c];
#pragma unroll
            for (int ww = 1; ww < kGemvWarps; ++ww) s += part[((size_t)ww * MT + m) * TILE + c];
            part[(size_t)m * TILE + c] = s;  // warp 0's slot: only this thread touches column c
        }
    }
    if (cn > 1) {
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
    const int chunk = TILE / (int)cn;  // this CTA finishes columns [rank * chunk, + chunk)
    __half *Y = static_cast<__half *>(a.Y);
    for (int idx = tid; idx < M * chunk; idx += THREADS) {
        const int m = idx / chunk, c = (int)rank * chunk + idx % chunk;
        const int n = tile * TILE + c;
        const float *src = part + (size_t)m * TILE + c;
        float s = 0.f;
        if (cn > 1) {
            for (unsigned r = 0; r < cn; ++r) s += ld_cluster(src, r);
        } else {
            s = *src;
        }
        if (n < N) Y[(int64_t)m * N + n] = __float2half_rn(s);
    }
    if (cn > 1) {  // no CTA leaves while another may read its partials
        cluster_arrive();
        cluster_wait();
    }
}

}  // namespace mt
