// pipe.cuh -- pipelined persistent backward for 16-byte-aligned rows (D % 8 == 0).
//
// Streaming. Each CTA is persistent and every thread streams ITS OWN 16-byte chunks
// of the next STAGES-1 rows into a shared-memory ring with cp.async (L2 only, no L1
// allocation), then reads them back for the current row. A thread only ever reads what
// it copied itself, so cp.async.wait_group alone orders the ring: no mbarrier, no
// cross-thread wait. Bytes in flight per SM are set by the ring depth (STAGES x streamed
// arrays x row slice), not by registers. A row split across a cluster exchanges its CTAs'
// row sums by the bounded push exchange of kernels.cuh; with a ring of three or more rows
// the exchange is software-pipelined (row j + 1's first pass runs while row j's sums are
// in flight). Before its grid-dependency wait, each CTA asks L2 for the rows its ring is
// first filled with (prefetch_l2, kernels.cuh).
//
// Ownership. Row assignment is static: CTA b runs row slots b*RPC + j*G*RPC
// (G = gridDim.x, j = 0, 1, ...), row group rg taking slot + rg. Thread t of a row group
// owns chunks k of EPC consecutive elements at columns (k*TPR + t)*EPC of every row it
// touches (EPC = 8, or 4 when every array is fp32; see PipeGeom); its dgamma/dbeta sums
// stay in fp32 registers across all its rows, and per-row statistics (rstd, mean) are
// prefetched into registers two rows ahead.
//
// Arithmetic. Blackwell executes fp32 pairs in one instruction (__ffma2_rn,
// __fmul2_rn, __fadd2_rn); the element math runs on float2 pairs, each lane rounded
// exactly as the scalar fp32 operation. When a thread's slice is small (CH <= 2) the
// converted row values and fp32 gamma (beta) stay in registers across the reduction
// barrier; for wider slices they are re-read from the ring and from per-thread
// parameter slots, which keeps the kernel free of register spills.
#pragma once

#include "kernels.cuh"

namespace mt {

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

// Shared-memory ring. Per stage and thread: CH chunks of X (UX 16-byte units each), of
// dY (UG units) and, with HAS_DS, of dS (UG units); after the STAGES stages, NPAR
// parameter slots of CH chunks of gamma (UW units). Unit u of a thread's chunk sits
// THREADS units after unit u-1, and consecutive threads own consecutive 16-byte words,
// so every ring access is bank-conflict free. Array ids: 0 = X, 1 = dY, 2 = dS.
template <int STAGES, int CH, int THREADS, int UX, int UG, bool HAS_DS, int UW, int NPAR>
struct Ring {
    static constexpr int kStageUnits = CH * (UX + UG * (HAS_DS ? 2 : 1));
    static constexpr size_t kStageBytes = (size_t)kStageUnits * THREADS * 16;
    static constexpr size_t kParamBytes = (size_t)NPAR * CH * UW * THREADS * 16;
    static constexpr size_t kBytes = STAGES * kStageBytes + kParamBytes;
    __device__ static __forceinline__ int index(int slot, int arr, int k, int tid) {
        const int base = (arr == 0) ? k * UX : (arr == 1) ? CH * UX + k * UG : CH * (UX + UG) + k * UG;
        return (slot * kStageUnits + base) * THREADS + tid;
    }
    __device__ static __forceinline__ int param(int k, int tid) {
        return (STAGES * kStageUnits + k * UW) * THREADS + tid;
    }
};

// Copy one chunk of type DT (chunk_units<DT, PPC>() 16-byte units) from global memory
// into ring units dst, dst + THREADS, ...
template <int DT, int PPC, int THREADS>
__device__ __forceinline__ void cp_chunk(uint4 *dst, const void *src) {
#pragma unroll
    for (int u = 0; u < chunk_units<DT, PPC>(); ++u)
        cp_async16(smem_addr(dst + u * THREADS), static_cast<const char *>(src) + 16 * u);
}

// Chunk geometry of a backward kernel. CH in the shape tables counts 8-element chunks.
// When every array is fp32 the kernel works in 4-element chunks (PPC = 2 pairs, CK = 2 CH
// of them), so each copy instruction of a warp covers 512 contiguous bytes; otherwise a
// chunk is 8 elements (PPC = 4, CK = CH) and an fp32 array's chunk takes two units.
template <int CH, int XT, int WT, int GT>
struct PipeGeom {
    static constexpr int PPC = (XT == kF32 && WT == kF32 && GT == kF32) ? 2 : 4;
    static constexpr int EPC = 2 * PPC;      // elements per chunk
    static constexpr int CK = CH * 4 / PPC;  // chunks per thread
    static constexpr int UX = chunk_units<XT, PPC>();
    static constexpr int UG = chunk_units<GT, PPC>();
    static constexpr int UW = chunk_units<WT, PPC>();
};

// Copy this thread's chunks of the parameter columns [beg, end) into its ring parameter
// slots.
template <class R, int WT, int PPC, int CK, int TPR, int THREADS>
__device__ __forceinline__ void stage_param(uint4 *ring, const void *src, int beg, int end, int t,
                                            int tid) {
#pragma unroll
    for (int k = 0; k < CK; ++k) {
        const int col = beg + (k * TPR + t) * 2 * PPC;
        if (col < end) cp_chunk<WT, PPC, THREADS>(&ring[R::param(k, tid)], as<WT>(src) + col);
    }
}

// Iterations every row group of row owner `owner` (of `owners`) runs (uniform across the
// CTA, and across a cluster that splits its rows).
__device__ __forceinline__ int owner_iterations(int64_t N, int rpc, int64_t owner, int64_t owners) {
    const int64_t base = owner * rpc;
    const int64_t stride = owners * rpc;
    return base < N ? (int)((N - base + stride - 1) / stride) : 0;
}

// ---------------------------------------------------------------- backward ---
// Dynamic shared memory: the ring (and gamma when CH > 2); after the row loop the ring
// is reused for the fixed-order combine of the CTA's row groups (NV x D floats).
// Compiled for CTAS resident CTAs per SM (it caps the registers per thread). X (or S) and
// dX are of type XT, gamma of type WT, dY and dS of type GT. CLU: rows split across a
// cluster (kernels.cuh, "cluster split"); the cluster is the row owner and writes one
// partial row, each CTA its slice of it.
// DSD (split rows of the fused op, fp16 dS): dS is loaded straight into registers at the
// start of its row's iteration instead of through the ring, so that the ring holds two
// arrays, is three deep and the exchange can be pipelined.
template <int OP, int TPR, int RPC, int CH, int STAGES, bool HAS_DS, int CTAS, int XT, int WT,
          int GT, bool CLU = false, bool DSD = false>
__global__ void __launch_bounds__(TPR * RPC, CTAS)
norm_bwd_pipe_kernel(const BwdArgs a) {
    constexpr int THREADS = TPR * RPC;
    constexpr int WPR = TPR / 32;
    constexpr int NV = (OP == kLayer) ? 2 : 1;
    constexpr bool KEEP = CH <= 2;
    using G = PipeGeom<CH, XT, WT, GT>;
    constexpr int PPC = G::PPC, EPC = G::EPC, CK = G::CK;
    constexpr bool DSR = HAS_DS && !DSD;  // dS through the ring
    using R = Ring<STAGES, CK, THREADS, G::UX, G::UG, DSR, G::UW, KEEP ? 0 : 1>;
    static_assert(TPR % 32 == 0 && THREADS <= 1024, "bad launch shape");
    static_assert(!CLU || RPC == 1, "a split row is one row group per CTA");
    // (the push exchange relies on the CTA barrier inside row_sum: TPR > 32)
    static_assert(!CLU || TPR > 32, "a split row's row group spans several warps");
    // Split rows with a ring of STAGES >= 3 software-pipeline the exchange (row j + 1's first
    // pass and push run before row j's collect); both passes then read the row from the ring
    // (gamma from registers when KEEP, else from the ring).
    constexpr bool PIPEX = CLU && STAGES >= 3;
    constexpr int NB = PIPEX ? 4 : 2;  // exchange buffers (kernels.cuh, cluster_collect)
    static_assert(!DSD || (PIPEX && HAS_DS && G::UG == 1), "dS in registers: pipelined split rows, 2-byte dS");
    __shared__ float red[2 * RPC * WPR * NV];
    extern __shared__ __align__(16) uint4 ring[];

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const float inv_d = 1.0f / (float)D;
    const Window<CLU> win(D, a.slice);
    const unsigned rank = CLU ? cluster_rank() : 0u;
    if constexpr (CLU) cluster_push_init(push_exchange<NB>());
    bool live = true;  // split rows: no wait of this thread has given up

    const int64_t owner = win.owner(), owners = win.owners();
    const int64_t stride = owners * RPC;
    const int64_t first = owner * RPC + rg;
    const int iters = owner_iterations(a.N, RPC, owner, owners);
    // L2 warm-up of the rows the ring is first filled with (kernels.cuh, prefetch_l2)
#pragma unroll
    for (int j = 0; j < STAGES - 1; ++j) {
        const int64_t row = first + (int64_t)j * stride;
        if (j < iters && row < a.N) {
            const int64_t off = row * (int64_t)D + win.beg;
            prefetch_l2(as<XT>(a.X) + off, win.end - win.beg, t, TPR);
            prefetch_l2(as<GT>(a.dY) + off, win.end - win.beg, t, TPR);
            if constexpr (HAS_DS) prefetch_l2(as<GT>(a.dS) + off, win.end - win.beg, t, TPR);
        }
    }

    pdl_enter();  // the dependent parameter reduction launches now and waits for this grid

    float2 gam[KEEP ? CK : 1][PPC];
    if constexpr (KEEP) {
#pragma unroll
        for (int k = 0; k < CK; ++k) {
            const int col = win.beg + (k * TPR + t) * EPC;
            ld_chunk<WT, kReadOnly, PPC>(as<WT>(a.gamma) + col, col < win.end, gam[k]);
        }
    } else {
        stage_param<R, WT, PPC, CK, TPR, THREADS>(ring, a.gamma, win.beg, win.end, t, tid);
    }
    cp_async_commit();

    float2 accg[CK][PPC];
    float2 accb[CK][(OP == kLayer) ? PPC : 1];
#pragma unroll
    for (int k = 0; k < CK; ++k) {
#pragma unroll
        for (int p = 0; p < PPC; ++p) accg[k][p] = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < ((OP == kLayer) ? PPC : 1); ++p) accb[k][p] = make_float2(0.f, 0.f);
    }

    auto issue = [&](int j) {
        const int64_t row = first + (int64_t)j * stride;
        if (j < iters && row < a.N) {
            const int slot = j % STAGES;
            const int64_t off = row * (int64_t)D;
#pragma unroll
            for (int k = 0; k < CK; ++k) {
                const int col = win.beg + (k * TPR + t) * EPC;
                if (col < win.end) {
                    cp_chunk<XT, PPC, THREADS>(&ring[R::index(slot, 0, k, tid)], as<XT>(a.X) + off + col);
                    cp_chunk<GT, PPC, THREADS>(&ring[R::index(slot, 1, k, tid)], as<GT>(a.dY) + off + col);
                    if constexpr (DSR)
                        cp_chunk<GT, PPC, THREADS>(&ring[R::index(slot, 2, k, tid)], as<GT>(a.dS) + off + col);
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

#pragma unroll
    for (int j = 0; j < STAGES - 1; ++j) issue(j);
    float r0, m0, r1, m1;
    stats(0, r0, m0);
    stats(1, r1, m1);

    if constexpr (PIPEX) {
        // Split rows, software-pipelined: iteration j runs row j + 1's first pass, CTA
        // reduction and push, then collects row j's cluster totals and runs row j's second
        // pass, so the exchange of row j is in flight while row j + 1 is read. The ring
        // holds rows j and j + 1 while row j + 2 loads (STAGES >= 3); a thread reads back
        // only the chunks it copied itself, so the ring needs no barrier.
        auto pass1 = [&](int j, float mu, float (&vv)[NV]) {
            const int slot = j % STAGES;
            const float2 nmu = make_float2(-mu, -mu);
            float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < CK; ++k) {
                if (win.beg + (k * TPR + t) * EPC >= win.end) continue;
                float2 xk[PPC], dk[PPC], g[PPC];
                unpack_chunk<XT, PPC>(&ring[R::index(slot, 0, k, tid)], THREADS, xk);
                unpack_chunk<GT, PPC>(&ring[R::index(slot, 1, k, tid)], THREADS, dk);
                if constexpr (KEEP) {
#pragma unroll
                    for (int p = 0; p < PPC; ++p) g[p] = gam[k][p];
                } else {
                    unpack_chunk<WT, PPC>(&ring[R::param(k, tid)], THREADS, g);
                }
#pragma unroll
                for (int p = 0; p < PPC; ++p) {
                    if constexpr (OP == kLayer) xk[p] = __fadd2_rn(xk[p], nmu);
                    const float2 gg = __fmul2_rn(dk[p], g[p]);
                    v0 = __ffma2_rn(gg, xk[p], v0);
                    if constexpr (OP == kLayer) v1 = __fadd2_rn(v1, gg);
                }
            }
            vv[0] = v0.x + v0.y;
            if constexpr (OP == kLayer) vv[NV - 1] = v1.x + v1.y;
        };
        auto pass2 = [&](int j, float r, float mu, const float (&vv)[NV], const uint4 (&dsr)[DSD ? CK : 1]) {
            const int slot = j % STAGES;
            const int64_t off = (first + (int64_t)j * stride) * (int64_t)D;
            const float c = r * vv[0] * inv_d;                           // mean_j g*xhat
            const float am = (OP == kLayer) ? vv[NV - 1] * inv_d : 0.f;  // mean_j g
            const float2 nmu = make_float2(-mu, -mu);
            const float2 r2 = make_float2(r, r);
            const float2 k2 = make_float2(-r * c, -r * c);
            const float2 ra2 = make_float2(-r * am, -r * am);
#pragma unroll
            for (int k = 0; k < CK; ++k) {
                const int col = win.beg + (k * TPR + t) * EPC;
                if (col >= win.end) continue;
                float2 xk[PPC], dk[PPC], g[PPC], o[PPC], sk[PPC];
                unpack_chunk<XT, PPC>(&ring[R::index(slot, 0, k, tid)], THREADS, xk);
                unpack_chunk<GT, PPC>(&ring[R::index(slot, 1, k, tid)], THREADS, dk);
                if constexpr (KEEP) {
#pragma unroll
                    for (int p = 0; p < PPC; ++p) g[p] = gam[k][p];
                } else {
                    unpack_chunk<WT, PPC>(&ring[R::param(k, tid)], THREADS, g);
                }
                if constexpr (DSD) unpack_chunk<GT, PPC>(&dsr[k], 1, sk);
                else if constexpr (HAS_DS) unpack_chunk<GT, PPC>(&ring[R::index(slot, 2, k, tid)], THREADS, sk);
#pragma unroll
                for (int p = 0; p < PPC; ++p) {
                    if constexpr (OP == kLayer) xk[p] = __fadd2_rn(xk[p], nmu);
                    const float2 xh = __fmul2_rn(xk[p], r2);
                    const float2 gg = __fmul2_rn(dk[p], g[p]);
                    const float2 base = (OP == kLayer) ? __ffma2_rn(gg, r2, ra2) : __fmul2_rn(gg, r2);
                    float2 dx = __ffma2_rn(xh, k2, base);
                    if constexpr (HAS_DS) dx = __fadd2_rn(dx, sk[p]);
                    o[p] = dx;
                    accg[k][p] = __ffma2_rn(dk[p], xh, accg[k][p]);
                    if constexpr (OP == kLayer) accb[k][p] = __fadd2_rn(accb[k][p], dk[p]);
                }
                st_chunk<XT, PPC>(as<XT>(a.dX) + off + col, o);
            }
        };
        PushExchange<NB> &px = push_exchange<NB>();
        // row 0: first pass and push (a split row's rows all exist: j < iters)
        float vc[NV];
        float rc = r0, mc = m0;
        if (iters > 0) {
            cp_async_wait<STAGES - 2>();
            pass1(0, mc, vc);
            row_sum<TPR, RPC, NV, true>(vc, red, 0, rg, wir, lane);
            cluster_push<NB, NV>(vc, px, 0, win.cn, rank);
        }
        for (int j = 0; j < iters; ++j) {
            issue(j + STAGES - 1);  // into row j - 1's slot, read by this thread last iteration
            uint4 dsr[DSD ? CK : 1];  // row j's dS, used by its second pass at the end
            if constexpr (DSD) {
                const int64_t offd = (first + (int64_t)j * stride) * (int64_t)D;
#pragma unroll
                for (int k = 0; k < CK; ++k) {
                    const int col = win.beg + (k * TPR + t) * EPC;
                    dsr[k] = col < win.end ? ld_unit<kStream>(as<GT>(a.dS) + offd + col) : make_uint4(0, 0, 0, 0);
                }
            }
            const float rn = r1, mn = m1;  // row j + 1
            stats(j + 2, r1, m1);
            float vn[NV];
            if (j + 1 < iters) {  // the same for every CTA of the cluster
                cp_async_wait<STAGES - 2>();
                pass1(j + 1, mn, vn);
                row_sum<TPR, RPC, NV, true>(vn, red, (j + 1) & 1, rg, wir, lane);
                cluster_push<NB, NV>(vn, px, j + 1, win.cn, rank);
            }
            if (!cluster_collect<NB, NV>(vc, px, j, win.cn, rank, live) && live) {
                atomicOr(a.status, kErrClusterWait);
                live = false;
            }
            if (live) pass2(j, rc, mc, vc, dsr);
            rc = rn;
            mc = mn;
#pragma unroll
            for (int i = 0; i < NV; ++i) vc[i] = vn[i];
        }
    } else {
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
        const float2 nmu = make_float2(-mu, -mu);

        // chunk k's centred x (LayerNorm: x - mean) and dY as fp32 pairs
        auto load_xd = [&](int k, float2 (&xk)[PPC], float2 (&dk)[PPC]) {
            unpack_chunk<XT, PPC>(&ring[R::index(slot, 0, k, tid)], THREADS, xk);
            unpack_chunk<GT, PPC>(&ring[R::index(slot, 1, k, tid)], THREADS, dk);
            if constexpr (OP == kLayer) {
#pragma unroll
                for (int p = 0; p < PPC; ++p) xk[p] = __fadd2_rn(xk[p], nmu);
            }
        };
        float2 xs[KEEP ? CK : 1][PPC], ds[KEEP ? CK : 1][PPC];

        // pass 1: sum_j g*(x - mean) and, for LayerNorm, sum_j g   (g = dY*gamma);
        // rstd is applied after the reduction: sum_j g*xhat = rstd * sum_j g*(x - mean)
        float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < CK; ++k) {
            const bool v = ok && win.beg + (k * TPR + t) * EPC < win.end;
            float2 xk[PPC], dk[PPC], g[PPC];
            if (v) {
                load_xd(k, xk, dk);
            } else {
#pragma unroll
                for (int p = 0; p < PPC; ++p) xk[p] = dk[p] = make_float2(0.f, 0.f);
            }
            if constexpr (KEEP) {
#pragma unroll
                for (int p = 0; p < PPC; ++p) { xs[k][p] = xk[p]; ds[k][p] = dk[p]; g[p] = gam[k][p]; }
            } else {
                if (v) {
                    unpack_chunk<WT, PPC>(&ring[R::param(k, tid)], THREADS, g);
                } else {
#pragma unroll
                    for (int p = 0; p < PPC; ++p) g[p] = make_float2(0.f, 0.f);
                }
            }
#pragma unroll
            for (int p = 0; p < PPC; ++p) {
                const float2 gg = __fmul2_rn(dk[p], g[p]);
                v0 = __ffma2_rn(gg, xk[p], v0);
                if constexpr (OP == kLayer) v1 = __fadd2_rn(v1, gg);
            }
        }
        float vv[NV];
        vv[0] = v0.x + v0.y;
        if constexpr (OP == kLayer) vv[NV - 1] = v1.x + v1.y;
        row_sum<TPR, RPC, NV, true>(vv, red, buf, rg, wir, lane);
        if constexpr (CLU) {
            if (!cluster_push_sum<NV>(vv, push_exchange<2>(), j, win.cn, rank, live) && live) {
                atomicOr(a.status, kErrClusterWait);
                live = false;
            }
        }
        const float c = r * vv[0] * inv_d;                           // mean_j g*xhat
        const float am = (OP == kLayer) ? vv[NV - 1] * inv_d : 0.f;  // mean_j g
        if (!ok || !live) continue;

        // pass 2: dX = r*g - r*a - (r*c)*xhat (+ dS), xhat = (x - mean)*r, and the
        // parameter-gradient sums dgamma += dY*xhat, dbeta += dY
        const float2 r2 = make_float2(r, r);
        const float2 k2 = make_float2(-r * c, -r * c);
        const float2 ra2 = make_float2(-r * am, -r * am);
#pragma unroll
        for (int k = 0; k < CK; ++k) {
            const int col = win.beg + (k * TPR + t) * EPC;
            if (col >= win.end) continue;
            float2 xk[PPC], dk[PPC], g[PPC], o[PPC];
            if constexpr (KEEP) {
#pragma unroll
                for (int p = 0; p < PPC; ++p) { xk[p] = xs[k][p]; dk[p] = ds[k][p]; g[p] = gam[k][p]; }
            } else {
                load_xd(k, xk, dk);
                unpack_chunk<WT, PPC>(&ring[R::param(k, tid)], THREADS, g);
            }
            float2 sk[PPC];
            if constexpr (HAS_DS) unpack_chunk<GT, PPC>(&ring[R::index(slot, 2, k, tid)], THREADS, sk);
#pragma unroll
            for (int p = 0; p < PPC; ++p) {
                const float2 xh = __fmul2_rn(xk[p], r2);
                const float2 gg = __fmul2_rn(dk[p], g[p]);
                const float2 base = (OP == kLayer) ? __ffma2_rn(gg, r2, ra2) : __fmul2_rn(gg, r2);
                float2 dx = __ffma2_rn(xh, k2, base);
                if constexpr (HAS_DS) dx = __fadd2_rn(dx, sk[p]);
                o[p] = dx;
                accg[k][p] = __ffma2_rn(dk[p], xh, accg[k][p]);
                if constexpr (OP == kLayer) accb[k][p] = __fadd2_rn(accb[k][p], dk[p]);
            }
            st_chunk<XT, PPC>(as<XT>(a.dX) + off + col, o);
        }
    }
    }  // (not PIPEX)
    cp_async_wait<0>();
    // split rows: this CTA's pushes are issued; no CTA leaves before the cluster's last
    // pushes into its buffers have landed (waited for below, after the partial rows)
    if constexpr (CLU) cluster_arrive();

    // Partials: the CTA's row groups are combined in the fixed order rg = 0, 1, ... and
    // one fp32 partial row per row owner (CTA, or cluster) is written.
    float *pg = a.part_g + (size_t)owner * D;
    float *pb = (OP == kLayer) ? a.part_b + (size_t)owner * D : nullptr;
    if constexpr (RPC == 1) {
#pragma unroll
        for (int k = 0; k < CK; ++k) {
            const int col = win.beg + (k * TPR + t) * EPC;
            if (col >= win.end) continue;
            float4 *g4 = reinterpret_cast<float4 *>(pg + col);
#pragma unroll
            for (int q = 0; q < PPC / 2; ++q)
                g4[q] = make_float4(accg[k][2 * q].x, accg[k][2 * q].y, accg[k][2 * q + 1].x,
                                    accg[k][2 * q + 1].y);
            if constexpr (OP == kLayer) {
                float4 *b4 = reinterpret_cast<float4 *>(pb + col);
#pragma unroll
                for (int q = 0; q < PPC / 2; ++q)
                    b4[q] = make_float4(accb[k][2 * q].x, accb[k][2 * q].y, accb[k][2 * q + 1].x,
                                        accb[k][2 * q + 1].y);
            }
        }
        if constexpr (CLU) cluster_wait();
    } else {
        __syncthreads();  // every thread is done with the ring
        float2 *cg2 = reinterpret_cast<float2 *>(ring);
        float2 *cb2 = cg2 + D / 2;
        for (int j = 0; j < RPC; ++j) {
            if (rg == j) {
#pragma unroll
                for (int k = 0; k < CK; ++k) {
                    const int col = (k * TPR + t) * EPC;
                    if (col >= D) continue;
#pragma unroll
                    for (int p = 0; p < PPC; ++p) {
                        const int i = col / 2 + p;
                        const float2 sg = (j == 0) ? accg[k][p] : __fadd2_rn(cg2[i], accg[k][p]);
                        if (j == RPC - 1) reinterpret_cast<float2 *>(pg)[i] = sg; else cg2[i] = sg;
                        if constexpr (OP == kLayer) {
                            const float2 sb = (j == 0) ? accb[k][p] : __fadd2_rn(cb2[i], accb[k][p]);
                            if (j == RPC - 1) reinterpret_cast<float2 *>(pb)[i] = sb; else cb2[i] = sb;
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace mt
