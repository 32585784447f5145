// pipe.cuh -- pipelined persistent kernels for 16-byte-aligned rows (D % 8 == 0).
//
// The plain kernels of kernels.cuh hold only the current row in flight per thread, so
// when a CTA reduces, nothing of its next row is on its way from HBM. Here each CTA is
// persistent and every thread streams ITS OWN 16-byte chunks of the next STAGES-1 rows
// into a shared-memory ring with cp.async (L2-only, no L1 allocation), then reads them
// back for the current row. Because a thread only ever reads what it copied itself,
// cp.async.wait_group alone orders the ring: no mbarrier, no cross-thread wait, and no
// wait that depends on another thread or CTA. Bytes in flight per SM are bounded by the
// ring (STAGES x arrays x row width), not by registers.
//
// Row assignment is static: CTA b runs row slots b*RPC + j*G*RPC (G = gridDim.x,
// j = 0, 1, ...), row group rg taking slot + rg. Thread t of a row group owns chunks
// k = 0..CH-1 at columns (k*TPR + t)*8 .. +7 of every row it touches, so its gamma (and
// beta) chunks are copied once into its own shared-memory slots and its dgamma/dbeta
// sums stay in fp32 registers across all its rows. Row data is re-read from the ring
// in each pass instead of being held in registers across the reduction barrier, which
// keeps register use (and so spills) down at wide rows. Per-row statistics (rstd,
// mean) are prefetched into registers two rows ahead.
#pragma once

#include "kernels.cuh"

namespace mt {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte global -> shared async copy, cached in L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Streaming 16-byte store (evict-first in L2): outputs are not re-read by this kernel.
__device__ __forceinline__ void st_global_cs(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    Raw<8> r;
    r.v = u;
    unpack<8>(r, f);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    u.x = float2_to_half2_bits(f[0], f[1]);
    u.y = float2_to_half2_bits(f[2], f[3]);
    u.z = float2_to_half2_bits(f[4], f[5]);
    u.w = float2_to_half2_bits(f[6], f[7]);
    return u;
}

// Shared-memory ring: [STAGES][NARR][CH][THREADS] x 16 bytes. Consecutive threads own
// consecutive 16-byte words, so ring reads are bank-conflict free.
// After the ring come NPAR parameter arrays (gamma, beta) in the same per-thread layout.
template <int STAGES, int NARR, int CH, int THREADS, int NPAR>
struct Ring {
    static constexpr size_t kBytes = (size_t)(STAGES * NARR + NPAR) * CH * THREADS * 16;
    __device__ static __forceinline__ int index(int slot, int arr, int k, int tid) {
        return ((slot * NARR + arr) * CH + k) * THREADS + tid;
    }
    __device__ static __forceinline__ int param(int p, int k, int tid) {
        return ((STAGES * NARR + p) * CH + k) * THREADS + tid;
    }
};

// Copy this thread's chunks of a parameter vector into its ring parameter slots.
template <class R, int CH, int TPR>
__device__ __forceinline__ void stage_param(uint4 *ring, int p, const __half *src, int D, int t,
                                            int tid) {
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        if (col < D) cp_async16(smem_addr(&ring[R::param(p, k, tid)]), src + col);
    }
}

// Iterations every row group of this CTA runs (uniform across the CTA).
__device__ __forceinline__ int cta_iterations(int64_t N, int rpc) {
    const int64_t base = (int64_t)blockIdx.x * rpc;
    const int64_t stride = (int64_t)gridDim.x * rpc;
    return base < N ? (int)((N - base + stride - 1) / stride) : 0;
}

// ----------------------------------------------------------------- forward ---
template <int OP, int TPR, int RPC, int CH, int STAGES>
__global__ void __launch_bounds__(TPR * RPC, 1)
norm_fwd_pipe_kernel(const FwdArgs a) {
    constexpr int THREADS = TPR * RPC;
    constexpr int WPR = TPR / 32;
    constexpr int NARR = (OP == kAddRms) ? 2 : 1;
    constexpr int NPAR = (OP == kLayer) ? 2 : 1;
    using R = Ring<STAGES, NARR, CH, THREADS, NPAR>;
    static_assert(TPR % 32 == 0 && THREADS <= 1024, "bad launch shape");
    __shared__ float red[2 * RPC * WPR];
    extern __shared__ __align__(16) uint4 ring[];

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const int64_t stride = (int64_t)gridDim.x * RPC;
    const int64_t first = (int64_t)blockIdx.x * RPC + rg;
    const int iters = cta_iterations(a.N, RPC);

    auto issue = [&](int j) {
        const int64_t row = first + (int64_t)j * stride;
        if (j < iters && row < a.N) {
            const int slot = j % STAGES;
            const int64_t off = row * (int64_t)D;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const int col = (k * TPR + t) * 8;
                if (col < D) {
                    cp_async16(smem_addr(&ring[R::index(slot, 0, k, tid)]), a.X + off + col);
                    if constexpr (OP == kAddRms)
                        cp_async16(smem_addr(&ring[R::index(slot, 1, k, tid)]), a.R + off + col);
                }
            }
        }
        cp_async_commit();
    };

    // group 0: this thread's gamma (and beta) chunks; then the first STAGES-1 rows
    stage_param<R, CH, TPR>(ring, 0, a.gamma, D, t, tid);
    if constexpr (OP == kLayer) stage_param<R, CH, TPR>(ring, 1, a.beta, D, t, tid);
    cp_async_commit();
#pragma unroll
    for (int j = 0; j < STAGES - 1; ++j) issue(j);

    int buf = 0;
    for (int j = 0; j < iters; ++j) {
        issue(j + STAGES - 1);
        cp_async_wait<STAGES - 1>();
        const int64_t row = first + (int64_t)j * stride;
        const bool ok = row < a.N;
        const int slot = j % STAGES;
        const int64_t off = (ok ? row : 0) * (int64_t)D;

        // x (fused op: x + r in fp32) of chunk k, re-read from the ring in each phase
        auto load_x = [&](int k, float (&xk)[8]) {
            const bool v = ok && (k * TPR + t) * 8 < D;
            unpack8(v ? ring[R::index(slot, 0, k, tid)] : make_uint4(0, 0, 0, 0), xk);
            if constexpr (OP == kAddRms) {
                float res[8];
                unpack8(v ? ring[R::index(slot, 1, k, tid)] : make_uint4(0, 0, 0, 0), res);
#pragma unroll
                for (int e = 0; e < 8; ++e) xk[e] += res[e];
            }
        };

        float mu = 0.f;
        if constexpr (OP == kLayer) {
            float s[1] = {0.f};
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                float xk[8];
                load_x(k, xk);
#pragma unroll
                for (int e = 0; e < 8; ++e) s[0] += xk[e];
            }
            row_sum<TPR, RPC, 1>(s, red, buf, rg, wir, lane);
            buf ^= 1;
            mu = s[0] / (float)D;
        }
        float q[1] = {0.f};
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = (k * TPR + t) * 8;
            const bool v = ok && col < D;
            float xk[8];
            load_x(k, xk);
            if constexpr (OP == kAddRms) {
                if (v) st_global_cs(a.S + off + col, pack8(xk));
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                // LayerNorm: centred second moment (two-pass)
                const float d = (OP == kLayer) ? (v ? xk[e] - mu : 0.f) : xk[e];
                q[0] += d * d;
            }
        }
        row_sum<TPR, RPC, 1>(q, red, buf, rg, wir, lane);
        buf ^= 1;
        const float rs = rsqrtf(q[0] / (float)D + a.eps);
        if (!ok) continue;
        if (t == 0) {
            a.rstd[row] = rs;
            if constexpr (OP == kLayer) a.mean[row] = mu;
        }
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = (k * TPR + t) * 8;
            if (col >= D) continue;
            float xk[8], g[8], y[8];
            load_x(k, xk);
            unpack8(ring[R::param(0, k, tid)], g);
            if constexpr (OP == kLayer) {
                float b[8];
                unpack8(ring[R::param(1, k, tid)], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = (xk[e] - mu) * rs * g[e] + b[e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = xk[e] * rs * g[e];
            }
            st_global_cs(a.Y + off + col, pack8(y));
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------- backward ---
// Dynamic shared memory: the ring and gamma; after the row loop the ring is reused for
// the fixed-order combine of the CTA's row groups (NV x D floats, which it covers).
template <int OP, int TPR, int RPC, int CH, int STAGES, bool HAS_DS>
__global__ void __launch_bounds__(TPR * RPC, 1)
norm_bwd_pipe_kernel(const BwdArgs a) {
    constexpr int THREADS = TPR * RPC;
    constexpr int WPR = TPR / 32;
    constexpr int NV = (OP == kLayer) ? 2 : 1;
    constexpr int NARR = HAS_DS ? 3 : 2;
    using R = Ring<STAGES, NARR, CH, THREADS, 1>;
    static_assert(TPR % 32 == 0 && THREADS <= 1024, "bad launch shape");
    __shared__ float red[2 * RPC * WPR * NV];
    extern __shared__ __align__(16) uint4 ring[];

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const float inv_d = 1.0f / (float)D;
    const int64_t stride = (int64_t)gridDim.x * RPC;
    const int64_t first = (int64_t)blockIdx.x * RPC + rg;
    const int iters = cta_iterations(a.N, RPC);

    float accg[CH][8];
    float accb[CH][(OP == kLayer) ? 8 : 1];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
#pragma unroll
        for (int e = 0; e < 8; ++e) accg[k][e] = 0.f;
#pragma unroll
        for (int e = 0; e < ((OP == kLayer) ? 8 : 1); ++e) accb[k][e] = 0.f;
    }

    auto issue = [&](int j) {
        const int64_t row = first + (int64_t)j * stride;
        if (j < iters && row < a.N) {
            const int slot = j % STAGES;
            const int64_t off = row * (int64_t)D;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const int col = (k * TPR + t) * 8;
                if (col < D) {
                    cp_async16(smem_addr(&ring[R::index(slot, 0, k, tid)]), a.X + off + col);
                    cp_async16(smem_addr(&ring[R::index(slot, 1, k, tid)]), a.dY + off + col);
                    if constexpr (HAS_DS)
                        cp_async16(smem_addr(&ring[R::index(slot, 2, k, tid)]), a.dS + off + col);
                }
            }
        }
        cp_async_commit();
    };
    auto stats = [&](int j, float &r, float &mu) {
        const int64_t row = first + (int64_t)j * stride;
        const bool ok = j < iters && row < a.N;
        r = ok ? __ldg(a.rstd + row) : 0.f;
        mu = (OP == kLayer && ok) ? __ldg(a.mean + row) : 0.f;
    };

    stage_param<R, CH, TPR>(ring, 0, a.gamma, D, t, tid);
    cp_async_commit();
#pragma unroll
    for (int j = 0; j < STAGES - 1; ++j) issue(j);
    float r0, m0, r1, m1;
    stats(0, r0, m0);
    stats(1, r1, m1);

    int buf = 0;
    for (int j = 0; j < iters; ++j, buf ^= 1) {
        issue(j + STAGES - 1);
        const float r = r0, mu = m0;
        r0 = r1;
        m0 = m1;
        stats(j + 2, r1, m1);
        cp_async_wait<STAGES - 1>();
        const int64_t row = first + (int64_t)j * stride;
        const bool ok = row < a.N;
        const int slot = j % STAGES;
        const int64_t off = (ok ? row : 0) * (int64_t)D;

        // pass 1: sum_j g*xhat and, for LayerNorm, sum_j g   (g = dY*gamma)
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = 0.f;
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            if (!ok || (k * TPR + t) * 8 >= D) continue;
            float gm[8], xv[8], dv[8];
            unpack8(ring[R::param(0, k, tid)], gm);
            unpack8(ring[R::index(slot, 0, k, tid)], xv);
            unpack8(ring[R::index(slot, 1, k, tid)], dv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xh = (xv[e] - mu) * r;
                const float g = dv[e] * gm[e];
                v[0] += g * xh;
                if constexpr (OP == kLayer) v[NV - 1] += g;
            }
        }
        row_sum<TPR, RPC, NV>(v, red, buf, rg, wir, lane);
        const float c = v[0] * inv_d;
        const float am = (OP == kLayer) ? v[NV - 1] * inv_d : 0.f;
        if (!ok) continue;

        // pass 2: dX = r*(g - a - xhat*c) (+ dS), and the parameter-gradient sums
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = (k * TPR + t) * 8;
            if (col >= D) continue;
            float gm[8], xv[8], dv[8], o[8];
            unpack8(ring[R::param(0, k, tid)], gm);
            unpack8(ring[R::index(slot, 0, k, tid)], xv);
            unpack8(ring[R::index(slot, 1, k, tid)], dv);
            float ds[8];
            if constexpr (HAS_DS) unpack8(ring[R::index(slot, 2, k, tid)], ds);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xh = (xv[e] - mu) * r;
                const float g = dv[e] * gm[e];
                float dx = r * ((g - am) - xh * c);
                if constexpr (HAS_DS) dx += ds[e];
                o[e] = dx;
                accg[k][e] += dv[e] * xh;
                if constexpr (OP == kLayer) accb[k][e] += dv[e];
            }
            st_global_cs(a.dX + off + col, pack8(o));
        }
    }
    cp_async_wait<0>();

    // Fixed-order combine of the row groups (rg = 0, 1, ...), one partial row per CTA.
    float *pg = a.part_g + (size_t)blockIdx.x * D;
    float *pb = (OP == kLayer) ? a.part_b + (size_t)blockIdx.x * D : nullptr;
    if constexpr (RPC == 1) {
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = (k * TPR + t) * 8;
            if (col >= D) continue;
            float4 *g4 = reinterpret_cast<float4 *>(pg + col);
            g4[0] = make_float4(accg[k][0], accg[k][1], accg[k][2], accg[k][3]);
            g4[1] = make_float4(accg[k][4], accg[k][5], accg[k][6], accg[k][7]);
            if constexpr (OP == kLayer) {
                float4 *b4 = reinterpret_cast<float4 *>(pb + col);
                b4[0] = make_float4(accb[k][0], accb[k][1], accb[k][2], accb[k][3]);
                b4[1] = make_float4(accb[k][4], accb[k][5], accb[k][6], accb[k][7]);
            }
        }
    } else {
        __syncthreads();  // every thread is done with the ring
        float *cg = reinterpret_cast<float *>(ring);
        float *cb = cg + D;
        for (int j = 0; j < RPC; ++j) {
            if (rg == j) {
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const int col = (k * TPR + t) * 8;
                    if (col >= D) continue;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float sg = (j == 0) ? accg[k][e] : cg[col + e] + accg[k][e];
                        if (j == RPC - 1) pg[col + e] = sg; else cg[col + e] = sg;
                        if constexpr (OP == kLayer) {
                            const float sb = (j == 0) ? accb[k][e] : cb[col + e] + accb[k][e];
                            if (j == RPC - 1) pb[col + e] = sb; else cb[col + e] = sb;
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace mt
