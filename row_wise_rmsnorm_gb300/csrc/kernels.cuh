// kernels.cuh -- sm_103a kernels for row-wise normalization (RMSNorm, LayerNorm,
// fused residual-add + RMSNorm), forward and backward.
//
// The work is HBM-bound (a few flops per 2-byte element), so there are no tensor
// cores here; the design goal is to stream every byte exactly once:
//
//  * A row group of TPR threads (TPR = 32: one warp per row; TPR > 32: several warps
//    per row) owns one row at a time. Thread t owns CH chunks of VEC contiguous
//    elements, chunk k starting at column (k*TPR + t)*VEC, so a warp's loads of
//    chunk k are contiguous and coalesced (VEC = 8: one 16-byte load per chunk).
//  * The row stays in registers between the reduction and the apply, so X (and R,
//    dY, S) is read from HBM exactly once.
//  * Row reductions: warp butterfly (shfl.xor), then, when a row spans several
//    warps, one shared-memory slot per warp summed by every thread in a fixed
//    order. The butterfly leaves bitwise-identical sums on every lane, and every
//    order is fixed, so results are reproducible bit for bit.
//  * Backward: a persistent grid; CTA b takes row slots b, b + G, b + 2G, ... (a
//    static assignment). Each thread keeps its columns' dgamma (and dbeta) sums in
//    fp32 registers across its rows; at the end the CTA's row groups are combined in
//    a fixed order and one fp32 partial row per CTA is written. A second small
//    kernel sums the partials column by column in ascending CTA order. No atomics.
//  * Rows wider than 16384 columns: the aligned forward streams the row twice on one
//    CTA (norm_fwd_stream_kernel; the second read mostly hits L2); the backward and
//    the scalar forward run on a thread-block cluster (see "cluster split" below): the
//    same per-thread layout inside each CTA's column window, plus one exchange of the
//    CTAs' row sums through distributed shared memory.
//
// Formulas (page title, section): meTile "Kernel coverage and training scope",
// "Exact native normalization contract"; tensorcore "Training kernels",
// "RMSnorm -- Llama-style" and "LayerNorm -- standard".
#pragma once

#include <type_traits>

#include <cuda_runtime.h>
#include <stdint.h>

#include "dtype.cuh"

namespace mt {

enum NormOp : int { kRms = 0, kLayer = 1, kAddRms = 2 };

// Activations X, R, S, Y are stored as xdt, gamma/beta as wdt (DType codes). The vector
// kernels take the types as template parameters; the scalar fallback reads these fields.
struct FwdArgs {
    const void *X;        // [N, D]
    const void *R;        // [N, D] residual (fused op only)
    const void *gamma;    // [D]
    const void *beta;     // [D] (LayerNorm only)
    void *S;              // [N, D] residual sum out (fused op only)
    void *Y;              // [N, D]
    float *mean;          // [N] (LayerNorm only)
    float *rstd;          // [N]
    int64_t N;
    int D;
    float eps;
    int xdt, wdt;
    int slice;            // cluster-split kernels: columns per CTA (a multiple of 8)
    int ahead;            // rows of the launch's resident CTAs (the L2 warm-up distance; 0: none)
};

// X (or the saved S) and dX are stored as xdt, gamma as wdt, dY/dS as gdt.
struct BwdArgs {
    const void *X;        // [N, D]: X (RMSNorm, LayerNorm) or the saved S (fused op)
    const void *gamma;    // [D]
    const void *dY;       // [N, D]
    const void *dS;       // [N, D] or nullptr (fused op only)
    const float *mean;    // [N] (LayerNorm only)
    const float *rstd;    // [N]
    void *dX;             // [N, D]
    float *part_g;        // [P, D] dgamma partials, one row per CTA
    float *part_b;        // [P, D] dbeta partials (LayerNorm only)
    int64_t N;
    int D;
    int xdt, wdt, gdt;
    int slice;            // cluster-split kernels: columns per CTA (a multiple of 8)
    unsigned *status;     // split rows: error bits of bounded waits (device memory)
};

// ------------------------------------------------------------------ helpers ---

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Eight fp16 values (one 16-byte chunk) <-> four fp32 pairs (the fp16 case of
// unpack_unit / pack_unit).
__device__ __forceinline__ void unpack8x2(const uint4 &u, float2 (&f)[4]) { unpack_unit<kF16>(u, f); }
__device__ __forceinline__ uint4 pack8x2(const float2 (&f)[4]) { return pack_unit<kF16>(f); }

// Programmatic dependent launch. Every kernel of this library is launched with the
// programmatic-stream-serialization attribute, so it may be scheduled while the
// previous kernel in the stream is still finishing. It therefore waits
// (griddepcontrol.wait) until that kernel has completed and its writes are visible
// before touching global memory, and it lets the next kernel launch early
// (griddepcontrol.launch_dependents); that kernel performs the same wait. Without the
// launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 warm-up, issued before pdl_enter(): a CTA that becomes resident while the previous
// kernel in the stream is still finishing asks L2 for the first bytes it will read, so
// that DRAM works during that kernel's tail instead of idling. prefetch.global.L2 returns
// no data to the thread. Global memory is coherent at L2, so a line fetched here that the
// previous kernel then writes holds the written bytes when the loads after the wait read
// it: the prefetch changes timing only. Threads t = 0 .. n-1 cover the 128-byte lines of
// the n_elem elements at p.
template <typename T>
__device__ __forceinline__ void prefetch_l2(const T *p, int n_elem, int t, int n) {
    const char *c = reinterpret_cast<const char *>(p);
    const int64_t bytes = (int64_t)n_elem * (int64_t)sizeof(T);
    for (int64_t b = (int64_t)t * 128; b < bytes; b += (int64_t)n * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + b));
}
// The same for the row-in-registers forwards, with a trip count known at compile time:
// a row group of TPR threads whose threads own CH 8-element chunks each spans at most
// CH*8*sizeof(T)*TPR bytes, so thread t asks for lines t, t + TPR, ... of the row at p.
template <int TPR, int CH, typename T>
__device__ __forceinline__ void prefetch_l2_row(const T *p, int D, int t) {
    constexpr int kLines = (CH * 8 * (int)sizeof(T) + 127) / 128;  // per thread
    const char *c = reinterpret_cast<const char *>(p);
    const int bytes = D * (int)sizeof(T);
#pragma unroll
    for (int i = 0; i < kLines; ++i) {
        const int b = (i * TPR + t) * 128;
        if (b < bytes) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + b));
    }
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------ cluster split ---
// Rows wider than one CTA's slice run on a thread-block cluster: CTA r of the cluster
// owns columns [r * slice, min(D, (r + 1) * slice)) of the cluster's rows, with the
// same per-thread chunk layout inside its slice as a CTA that owns a whole row. A row
// reduction first sums within each CTA (row_sum), then cluster_sum adds the CTAs'
// totals through distributed shared memory in rank order 0, 1, ..., so every CTA of
// the cluster ends with the bitwise-identical row total. The cluster barrier is the
// hardware one (every CTA of a cluster is resident at once, so it always completes).

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_size() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Release this thread's earlier memory accesses to the cluster / wait for every thread
// of every CTA of the cluster to have arrived (acquiring their accesses).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The float at the same shared-memory offset as `local`, in the CTA of cluster rank r.
__device__ __forceinline__ float ld_cluster(const float *local, unsigned r) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(r));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Cluster-wide sum of NV per-CTA totals (every thread of the CTA holds them, bitwise
// identical). xch: 2 x NV shared floats; alternate `buf` between consecutive calls (a
// CTA rewrites a slot only after the next call's barrier, which every CTA reaches only
// once it has read the slot). Every thread of every CTA of the cluster must call it.
// After the barrier, lane r of every warp reads CTA r's totals (one distributed
// shared-memory load each) and a warp butterfly adds them: the same operands in the
// same lanes everywhere, so every thread of the cluster gets the same bits.
template <int NV>
__device__ __forceinline__ void cluster_sum(float (&v)[NV], float *xch, int buf, unsigned n) {
    float *slot = xch + buf * NV;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) slot[i] = v[i];
    }
    cluster_arrive();
    cluster_wait();
    const unsigned lane = threadIdx.x & 31u;
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = warp_sum(lane < n ? ld_cluster(slot + i, lane) : 0.f);
}

// LayerNorm statistics of a split row in one exchange. Each CTA has the sum s and the
// centred second moment m2 (about its own slice mean) of its n columns. With the row
// mean mu = (sum of the s) / D, the row's centred sum of squares is exactly
//   sum over slices of ( m2 + n (s/n - mu)^2 )
// (within-slice plus between-slice parts; Chan, Golub and LeVeque, "Algorithms for
// computing the sample variance: analysis and recommendations", 1983), as stable as the
// two-pass form since every term is a sum of squares about a mean. xch: 4 shared floats
// (2 buffers of {s, m2}); v = {s, m2} in, {row mean, row centred sum of squares} out.
// Same calling rules and lane-parallel combination as cluster_sum.
__device__ __forceinline__ void cluster_ln_stats(float (&v)[2], float *xch, int buf, unsigned n,
                                                 int D, int slice) {
    float *slot = xch + buf * 2;
    if (threadIdx.x == 0) {
        slot[0] = v[0];
        slot[1] = v[1];
    }
    cluster_arrive();
    cluster_wait();
    const unsigned lane = threadIdx.x & 31u;
    float sr = 0.f, m2r = 0.f, nr = 0.f;
    if (lane < n) {
        const int beg = (int)lane * slice;
        nr = (float)max(0, min(D, beg + slice) - beg);
        sr = ld_cluster(slot, lane);
        m2r = ld_cluster(slot + 1, lane);
    }
    const float mu = warp_sum(sr) / (float)D;
    const float dev = nr > 0.f ? sr / nr - mu : 0.f;
    v[0] = mu;
    v[1] = warp_sum(m2r + nr * dev * dev);
}

// ------------------------------------------------------ push exchange ---
// The pipelined backward of a split row exchanges its CTAs' row sums by pushing them
// instead of meeting at the cluster barrier: after its CTA-level reduction, thread 0 of
// every CTA writes the CTA's totals (two floats) into its slot of each peer's buffer with
// st.async, an asynchronous store into distributed shared memory that completes 8 bytes
// of transactions on the peer's mbarrier, and arrives on its own mbarrier expecting
// (cn - 1) * 8 bytes. Each CTA waits only on its own mbarrier until its peers' totals are
// in, and adds the cn totals in rank order (every CTA the same operands in the same
// order: the same bits). A CTA waits for data, not for its peers to reach a barrier, and
// no store is fenced.
// Two buffers alternate by row. A CTA pushes row j + 2 into the buffer of row j only
// after receiving every peer's row j + 1 totals, which each peer pushed after all its
// threads had passed the row j wait and read the row j buffer (a CTA barrier lies
// between), so a buffer is never overwritten before it is read and no transaction of
// row j + 2 can land in the phase of row j.
//
// Every wait is bounded (kWaitLimitNs of global time): a wait that gives up ORs
// kErrClusterWait into the launch's status word (read on the host with
// mt_device_wait_errors), and the thread skips its remaining waits; the kernel runs to
// its end, so no wait can hang the GPU.
constexpr unsigned kErrClusterWait = 1u;
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;  // 200 ms
constexpr int kMaxPushCluster = 16;

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes this thread's mbarrier initialisations visible across the cluster.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive on this CTA's mbarrier and add `bytes` to the phase's expected transactions.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// True once the phase with parity `parity` of the local mbarrier has completed (acquire at
// cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, unsigned parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// mbar_try_wait_cluster until it succeeds or kWaitLimitNs have passed (then false).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, unsigned parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_cluster(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// The shared::cluster address of `local`'s counterpart in the CTA of cluster rank r.
__device__ __forceinline__ uint32_t cluster_map(const void *local, unsigned r) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(r));
    return remote;
}

// Store two floats at `addr` (another CTA's shared memory, 8-byte aligned), completing 8
// bytes of transactions on that CTA's mbarrier at `bar`.
__device__ __forceinline__ void st_async_f2(uint32_t addr, float x, float y, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
        ::"r"(addr), "f"(x), "f"(y), "r"(bar)
        : "memory");
}

// NB row buffers, used by rows j with j % NB = buffer (parity of the buffer's mbarrier
// phase: (j / NB) & 1). NB = 2 when a CTA waits for row j's totals before it pushes row
// j + 1; NB = 4 when it pushes row j + 1 before it waits for row j (the software-pipelined
// backward, whose safety argument is at cluster_collect).
template <int NB>
struct PushExchange {
    uint64_t bar[NB];                           // one per row buffer
    __align__(8) float in[NB][kMaxPushCluster][2];  // [buffer][rank of the sender][value]
};

// The exchange state of this CTA (static shared memory of the kernels that call it only).
template <int NB>
__device__ __forceinline__ PushExchange<NB> &push_exchange() {
    __shared__ __align__(8) PushExchange<NB> px;
    return px;
}

// Thread 0 initialises the exchange; every thread of every CTA of the cluster must then
// pass one cluster barrier before the first push (cluster_push_init does both).
template <int NB>
__device__ __forceinline__ void cluster_push_init(PushExchange<NB> &px) {
    if (threadIdx.x == 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) mbar_init(&px.bar[b], 1);
        mbar_init_fence();
    }
    cluster_arrive();
    cluster_wait();
}

// Push this CTA's NV (1 or 2) totals of the cluster's j-th row (bitwise identical in every
// thread of the CTA) into every peer's buffer j % NB, and arrive on the CTA's own barrier
// of that buffer expecting the peers' (cn - 1) pushes. Thread 0 does the work.
template <int NB, int NV>
__device__ __forceinline__ void cluster_push(const float (&v)[NV], PushExchange<NB> &px, int j,
                                             unsigned cn, unsigned rank) {
    static_assert(NV == 1 || NV == 2, "one or two values per row");
    const int buf = j % NB;
    if (threadIdx.x == 0) {
        const float y = (NV == 2) ? v[NV - 1] : 0.f;
        for (unsigned r = 0; r < cn; ++r) {
            if (r == rank) continue;
            st_async_f2(cluster_map(&px.in[buf][rank][0], r), v[0], y,
                        cluster_map(&px.bar[buf], r));
        }
        mbar_arrive_expect_tx(&px.bar[buf], (cn - 1) * 8u);
    }
}

// Wait (bounded) until every peer's totals of row j are in buffer j % NB, then replace v
// (this CTA's own totals of row j) by the cluster's sum in rank order 0, 1, ... (the same
// operands in the same order in every CTA: the same bits). `live`: this thread's waits have
// not given up so far; returns false if this wait gave up (the totals are incomplete).
//
// Buffer reuse. A CTA pushes row j into its peers' buffer j % NB, which last held row
// j - NB; a peer's threads read that row in their cluster_collect of row j - NB. With
// NB = 2 (push row j, then collect row j, each row in turn): a CTA pushes row j only after
// collecting row j - 1, whose pushes each peer made after all its threads had collected
// row j - 2 (a CTA barrier lies between). With NB = 4 and rows pipelined (push row j + 1,
// then collect row j): a CTA pushes row j + 1 only after collecting row j - 1, which each
// peer pushed in its iteration j - 2, after all its threads had collected row j - 3 in
// iteration j - 3 (a CTA barrier lies between), and row j - 3 is the row that buffer
// (j + 1) % 4 held. In both cases no push lands in a buffer before its previous row has
// been read, and no transaction of row j + NB reaches a barrier phase before the phase of
// row j has completed.
template <int NB, int NV>
__device__ __forceinline__ bool cluster_collect(float (&v)[NV], PushExchange<NB> &px, int j,
                                                unsigned cn, unsigned rank, bool live) {
    const int buf = j % NB;
    const bool ok = live && mbar_wait_cluster_bounded(&px.bar[buf], (unsigned)(j / NB) & 1u);
    float t[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) t[i] = 0.f;
    for (unsigned r = 0; r < cn; ++r)
#pragma unroll
        for (int i = 0; i < NV; ++i) t[i] += (r == rank) ? v[i] : px.in[buf][r][i];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = t[i];
    return ok;
}

// Cluster-wide sum of the NV per-CTA totals of the cluster's j-th row: push, then collect.
// Every thread of every CTA of the cluster calls it once per row, and between two calls
// every thread of the CTA passes a CTA barrier.
template <int NV>
__device__ __forceinline__ bool cluster_push_sum(float (&v)[NV], PushExchange<2> &px, int j,
                                                 unsigned cn, unsigned rank, bool live) {
    cluster_push<2, NV>(v, px, j, cn, rank);
    return cluster_collect<2, NV>(v, px, j, cn, rank, live);
}

// This CTA's column window and row owner. Not split: columns [0, D) and the plain CTA
// index. Split: the CTA's slice, and the cluster index as the owner (cn = cluster size).
template <bool CLU>
struct Window {
    int beg, end;
    unsigned cn;
    __device__ __forceinline__ Window(int D, int slice) {
        if constexpr (CLU) {
            cn = cluster_size();
            beg = (int)cluster_rank() * slice;
            end = min(D, beg + slice);
        } else {
            cn = 1;
            beg = 0;
            end = D;
        }
    }
    __device__ __forceinline__ int64_t owner() const {
        return CLU ? (int64_t)(blockIdx.x / cn) : (int64_t)blockIdx.x;
    }
    __device__ __forceinline__ int64_t owners() const {
        return CLU ? (int64_t)(gridDim.x / cn) : (int64_t)gridDim.x;
    }
};

// Barrier for one row group. NAMED: named barrier 1 + rg over the group's TPR threads,
// so the row groups of a CTA do not wait for one another (the persistent backward, where
// row groups run many rows; measured faster there). Otherwise, and for a CTA that is a
// single row group, barrier 0 (__syncthreads; measured faster in the forward, where
// every row group runs one row and exits).
template <int TPR, int RPC, bool NAMED>
__device__ __forceinline__ void row_group_sync(int rg) {
    if constexpr (RPC == 1 || !NAMED) {
        __syncthreads();
    } else {
        static_assert(RPC < 16, "one named barrier per row group");
        asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "n"(TPR) : "memory");
    }
}

// Sum NV values over the TPR threads of one row group. `red` holds
// 2 (buffers) x RPC x WPR x NV floats; alternate `buf` between consecutive calls so
// one barrier per call suffices. When WPR > 1 it contains a barrier (see row_group_sync):
// every thread of the row group (of the CTA, unless NAMED) must call it. Each warp first reduces with a
// butterfly; then lane l of every warp reads warp l's sum (zero for l >= WPR) and a
// second butterfly adds them. The operands and their order are the same in every
// warp, so every thread ends with the bitwise-identical total.
template <int TPR, int RPC, int NV, bool NAMED = false>
__device__ __forceinline__ void row_sum(float (&v)[NV], float *red, int buf, int rg, int wir,
                                        int lane) {
    constexpr int WPR = TPR / 32;
    static_assert(WPR <= 32, "row group wider than 32 warps");
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = warp_sum(v[i]);
    if constexpr (WPR > 1) {
        float *s = red + ((buf * RPC + rg) * WPR) * NV;
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NV; ++i) s[wir * NV + i] = v[i];
        }
        row_group_sync<TPR, RPC, NAMED>(rg);
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = warp_sum(lane < WPR ? s[lane * NV + i] : 0.f);
    }
}

// ------------------------------------------------------------------ forward ---
// Scalar fallback for any alignment and any width: one row group per row, thread t
// owning the CH columns k*TPR + t; types chosen at run time (a.xdt, a.wdt).
// grid = ceil(N / RPC) CTAs of TPR*RPC threads.
template <int OP, int TPR, int RPC, int CH, bool CLU = false>
__global__ void __launch_bounds__(TPR * RPC)
norm_fwd_kernel(const FwdArgs a) {
    pdl_enter();
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad launch shape");
    static_assert(!CLU || RPC == 1, "a split row is one row group per CTA");
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * RPC * WPR];
    __shared__ float xch[CLU ? 4 : 1];  // cluster_sum (2) or cluster_ln_stats (4)

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const Window<CLU> win(D, a.slice);
    const int64_t row = CLU ? win.owner() : (int64_t)blockIdx.x * RPC + rg;
    const bool ok = row < a.N;  // split rows: the grid is N clusters, so always true
    // A single-warp row group has no CTA barrier, so it may leave early; wider row
    // groups run masked (all loads read 0, nothing is stored) to reach the barriers.
    if (WPR == 1 && !ok) return;
    const int64_t off = (ok ? row : 0) * (int64_t)D;
    const int lim = ok ? win.end : 0;  // masked row: every column counts as past the end

    float x[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = win.beg + k * TPR + t;
        const bool v = col < lim;
        x[k] = v ? ld_elem_stream(a.X, off + col, a.xdt) : 0.f;
        if constexpr (OP == kAddRms) {
            // fused op: s = x + r in fp32, normalise the unrounded s, store s rounded
            x[k] += v ? ld_elem_stream(a.R, off + col, a.xdt) : 0.f;
            if (v) st_elem(a.S, off + col, x[k], a.xdt);
        }
    }

    // LayerNorm: the mean, then the centred second moment (two passes, from registers).
    // A split row centres on its slice's own mean and combines the slices afterwards.
    float mu = 0.f, s[1] = {0.f};
    if constexpr (OP == kLayer) {
#pragma unroll
        for (int k = 0; k < CH; ++k) s[0] += x[k];
        row_sum<TPR, RPC, 1>(s, red, 0, rg, wir, lane);
        mu = s[0] / (float)(CLU ? max(win.end - win.beg, 1) : D);
    }
    float q[1] = {0.f};
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const float d = (OP == kLayer) ? ((win.beg + k * TPR + t) < lim ? x[k] - mu : 0.f) : x[k];
        q[0] += d * d;
    }
    row_sum<TPR, RPC, 1>(q, red, 1, rg, wir, lane);
    if constexpr (CLU) {
        if constexpr (OP == kLayer) {
            float v[2] = {s[0], q[0]};
            cluster_ln_stats(v, xch, 0, win.cn, D, a.slice);
            mu = v[0];
            q[0] = v[1];
        } else {
            cluster_sum<1>(q, xch, 0, win.cn);
        }
        cluster_arrive();  // done reading the other CTAs' slots (waited for before exit)
    }
    const float rs = rsqrtf(q[0] / (float)D + a.eps);
    if (!ok) return;  // after the last barrier
    if (t == 0 && win.beg == 0) {
        a.rstd[row] = rs;
        if constexpr (OP == kLayer) a.mean[row] = mu;
    }

#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = win.beg + k * TPR + t;
        if (col >= win.end) continue;
        const float g = ld_elem(a.gamma, col, a.wdt);
        float y;
        if constexpr (OP == kLayer) y = (x[k] - mu) * rs * g + ld_elem(a.beta, col, a.wdt);
        else y = x[k] * rs * g;
        st_elem(a.Y, off + col, y, a.xdt);
    }
    if constexpr (CLU) cluster_wait();  // no CTA leaves while another may read its slots
}

// Forward for 16-byte-aligned rows (D % 8 == 0), one row group per row, fp32 pair
// arithmetic (__ffma2_rn & co.). Rows are loaded once with streaming loads and stay in
// registers (as fp32 pairs) through the reductions and the apply. Activations are of
// type XT, gamma/beta of type WT. MINB is the minimum number of resident CTAs per SM
// asked of the compiler (it bounds the registers per thread; 0: the compiler's choice).
template <int OP, int TPR, int RPC, int CH, int MINB, int XT, int WT>
__global__ void __launch_bounds__(TPR * RPC, MINB)
norm_fwd_vec8_kernel(const FwdArgs a) {
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad launch shape");
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * RPC * WPR];

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const float inv_d = 1.0f / (float)D;
    const int64_t row = (int64_t)blockIdx.x * RPC + rg;
    const bool ok = row < a.N;
    // (not at 16 CTAs of 128 threads: in 32 registers a thread its addresses spill)
    if (ok && MINB * TPR * RPC < 2048) {
        prefetch_l2_row<TPR, CH>(as<XT>(a.X) + row * (int64_t)D, D, t);
        if constexpr (OP == kAddRms) prefetch_l2_row<TPR, CH>(as<XT>(a.R) + row * (int64_t)D, D, t);
    }
    pdl_enter();
    if (WPR == 1 && !ok) return;  // no CTA barrier in a single-warp row group
    const int64_t off = (ok ? row : 0) * (int64_t)D;

    float2 x[CH][4];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        const bool v = ok && col < D;
        ld_chunk<XT, kStream>(as<XT>(a.X) + off + col, v, x[k]);
        if constexpr (OP == kAddRms) {
            float2 r[4];
            ld_chunk<XT, kStream>(as<XT>(a.R) + off + col, v, r);
#pragma unroll
            for (int p = 0; p < 4; ++p) x[k][p] = __fadd2_rn(x[k][p], r[p]);
            if (v) st_chunk<XT>(as<XT>(a.S) + off + col, x[k]);
        }
    }
    // LayerNorm: the mean, then the centred second moment (two passes, from registers).
    float mu = 0.f, s[1] = {0.f};
    if constexpr (OP == kLayer) {
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < CH; ++k)
#pragma unroll
            for (int p = 0; p < 4; ++p) s2 = __fadd2_rn(s2, x[k][p]);
        s[0] = s2.x + s2.y;
        row_sum<TPR, RPC, 1>(s, red, 0, rg, wir, lane);
        mu = s[0] * inv_d;
    }
    float2 nmu = make_float2(-mu, -mu);
    float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        if (!(ok && (k * TPR + t) * 8 < D)) continue;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 d = (OP == kLayer) ? __fadd2_rn(x[k][p], nmu) : x[k][p];
            q2 = __ffma2_rn(d, d, q2);
        }
    }
    float q[1] = {q2.x + q2.y};
    row_sum<TPR, RPC, 1>(q, red, 1, rg, wir, lane);
    const float rs = rsqrtf(q[0] * inv_d + a.eps);
    if (!ok) return;  // after the last barrier
    if (t == 0) {
        a.rstd[row] = rs;
        if constexpr (OP == kLayer) a.mean[row] = mu;
    }
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        if (col >= D) continue;
        float2 g[4], y[4];
        ld_param<WT>(as<WT>(a.gamma) + col, g);
        if constexpr (OP == kLayer) {
            float2 b[4];
            ld_param<WT>(as<WT>(a.beta) + col, b);
#pragma unroll
            for (int p = 0; p < 4; ++p)
                y[p] = __ffma2_rn(__fmul2_rn(__fadd2_rn(x[k][p], nmu), rs2), g[p], b[p]);
        } else {
#pragma unroll
            for (int p = 0; p < 4; ++p) y[p] = __fmul2_rn(__fmul2_rn(x[k][p], rs2), g[p]);
        }
        st_chunk<XT>(as<XT>(a.Y) + off + col, y);
    }
}

// The same forward for RMSNorm and LayerNorm with 2-byte activations (XT = fp16 or
// bf16), the row kept as the loaded 16-byte chunks and widened to fp32 pairs at each use:
// half the registers of norm_fwd_vec8_kernel, so more CTAs (and more bytes in flight)
// fit per SM, for one more conversion per pass. (The fused op normalises the unrounded
// fp32 x + r, so it cannot keep 2-byte chunks.)
template <int OP, int TPR, int RPC, int CH, int MINB, int XT, int WT>
__global__ void __launch_bounds__(TPR * RPC, MINB)
norm_fwd_packed_kernel(const FwdArgs a) {
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad launch shape");
    static_assert(OP == kRms || OP == kLayer, "the fused op keeps its fp32 sum");
    static_assert(XT == kF16 || XT == kBF16, "2-byte activations only");
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * RPC * WPR];
    const auto *X = as<XT>(a.X);

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const float inv_d = 1.0f / (float)D;
    const int64_t row = (int64_t)blockIdx.x * RPC + rg;
    const bool ok = row < a.N;
    if (ok) prefetch_l2_row<TPR, CH>(X + row * (int64_t)D, D, t);
    pdl_enter();
    if (WPR == 1 && !ok) return;  // no CTA barrier in a single-warp row group
    const int64_t off = (ok ? row : 0) * (int64_t)D;

    uint4 raw[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        raw[k] = (ok && col < D) ? ld_unit<kStream>(X + off + col) : make_uint4(0, 0, 0, 0);
    }
    // RMSNorm: with its row's loads issued, thread 0 of the row group warms L2 with the row
    // the next wave takes, `ahead` rows on (one bulk prefetch). Measured on GB300: RMSNorm
    // 16384 x 4096 forward 40.2 -> 39.2 us, 8192 x 8192 40.3 -> 39.2 us; LayerNorm lost
    // (2048 x 16384 22.7 -> 23.7 us), so it does not prefetch.
    if constexpr (OP == kRms) {
        if (t == 0 && ok && a.ahead > 0 && row + a.ahead < a.N)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(X + (row + a.ahead) * (int64_t)D),
                         "r"((unsigned)D * (unsigned)sizeof(*X)) : "memory");
    }
    // Chunk k as fp32 pairs. Each pass widens the chunks again rather than keep fp32
    // copies of the row alive across the reductions. So that the compiler does not merge
    // those conversions, a pass XORs the words with `zero & bits(after)`, where `after`
    // is a value of that pass (the mean, rstd) and `zero` is a runtime zero (D < 2^30):
    // the words are unchanged, but each pass's conversions have their own inputs, which
    // exist only once the pass's reduction is done.
    const uint32_t zero = (uint32_t)D >> 30;
    auto pairs = [&](int k, float2 (&f)[4], float after) {
        const uint32_t key = zero & __float_as_uint(after);
        unpack_unit<XT>(make_uint4(raw[k].x ^ key, raw[k].y ^ key, raw[k].z ^ key, raw[k].w ^ key), f);
    };

    // LayerNorm: as in norm_fwd_vec8_kernel
    float mu = 0.f, s[1] = {0.f};
    if constexpr (OP == kLayer) {
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            float2 f[4];
            unpack_unit<XT>(raw[k], f);
#pragma unroll
            for (int p = 0; p < 4; ++p) s2 = __fadd2_rn(s2, f[p]);
        }
        s[0] = s2.x + s2.y;
        row_sum<TPR, RPC, 1>(s, red, 0, rg, wir, lane);
        mu = s[0] * inv_d;
    }
    float2 nmu = make_float2(-mu, -mu);
    float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        if (!(ok && (k * TPR + t) * 8 < D)) continue;
        float2 f[4];
        if constexpr (OP == kLayer) pairs(k, f, mu);
        else unpack_unit<XT>(raw[k], f);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 d = (OP == kLayer) ? __fadd2_rn(f[p], nmu) : f[p];
            q2 = __ffma2_rn(d, d, q2);
        }
    }
    float q[1] = {q2.x + q2.y};
    row_sum<TPR, RPC, 1>(q, red, 1, rg, wir, lane);
    const float rs = rsqrtf(q[0] * inv_d + a.eps);
    if (!ok) return;  // after the last barrier
    if (t == 0) {
        a.rstd[row] = rs;
        if constexpr (OP == kLayer) a.mean[row] = mu;
    }
    const float2 rs2 = make_float2(rs, rs);
    // gamma (beta) are read chunk by chunk at the point of use: `chain` (always zero)
    // makes each chunk's parameter address depend on rs and on the previous chunk's
    // result, so the compiler neither hoists the loads above the reductions nor issues
    // all chunks' loads at once, either of which would hold CH x 16 (32) bytes of
    // registers per thread.
    uint32_t chain = zero & __float_as_uint(rs);
#pragma unroll
    for (int k = 0; k < CH; ++k) {
        const int col = (k * TPR + t) * 8;
        if (col >= D) continue;
        float2 f[4], g[4], y[4];
        pairs(k, f, rs);
        const int pc = col + (int)chain;
        ld_param<WT>(as<WT>(a.gamma) + pc, g);
        if constexpr (OP == kLayer) {
            float2 b[4];
            ld_param<WT>(as<WT>(a.beta) + pc, b);
#pragma unroll
            for (int p = 0; p < 4; ++p)
                y[p] = __ffma2_rn(__fmul2_rn(__fadd2_rn(f[p], nmu), rs2), g[p], b[p]);
        } else {
#pragma unroll
            for (int p = 0; p < 4; ++p) y[p] = __fmul2_rn(__fmul2_rn(f[p], rs2), g[p]);
        }
        chain = zero & __float_as_uint(y[0].x);
        st_chunk<XT>(as<XT>(a.Y) + off + col, y);
    }
}

// --------------------------------------------------- wide rows, streamed ---
// Chunks in flight per thread for the streaming kernels: a table's UN counts 16-byte
// chunks of a 2-byte type; fp32 chunks are 32 bytes, so fp32 rows take half as many.
__host__ __device__ constexpr int stream_un(int xt, int un) { return xt == kF32 ? (un + 1) / 2 : un; }

// Forward for aligned rows wider than a CTA holds in registers (D > 16384): one CTA of
// TPR threads per row, two passes over the row; chunk c (8 elements) belongs to thread
// c % TPR, UN chunks in flight per thread and operand. Pass 1 reads the row with the
// default cache policy (so pass 2 mostly finds it in L2; the fused op also writes S) and
// reduces it: RMSNorm and the fused op the sum of squares; LayerNorm, per thread, the
// count, sum and centred sum of squares of its elements, one batch of UN chunks at a time
// (each batch centred on its own mean, then merged by the update of Chan, Golub and
// LeVeque), and the row's centred sum of squares as sum_t (m2_t + n_t (s_t / n_t - mu)^2).
// LayerNorm works on x - k, k the row's first element, so that every mean in these sums
// is of the row's spread, not of its offset from zero: a row with mean 1000 and standard
// deviation 0.1 keeps its variance digits, and the apply takes (x - k) - mean(x - k),
// so its outputs keep theirs too. Pass 2 reads the row again (the fused op re-adds
// x + r, the same fp32 value as pass 1) and applies. MINB: resident CTAs per SM asked of the
// compiler (a register cap).
constexpr int64_t kStreamAheadBytes = 128 * 1024;

template <int OP, int TPR, int UN, int MINB, int XT, int WT>
__global__ void __launch_bounds__(TPR, MINB)
norm_fwd_stream_kernel(const FwdArgs a) {
    static_assert(TPR % 32 == 0 && TPR <= 1024, "bad launch shape");
    constexpr int WPR = TPR / 32;
    __shared__ float red[2 * WPR];
    const int t = threadIdx.x, wir = t / 32, lane = t % 32;
    const int D = a.D;
    const float inv_d = 1.0f / (float)D;
    const int64_t row = blockIdx.x;
    const int64_t off = row * (int64_t)D;
    prefetch_l2(as<XT>(a.X) + off, min(D, UN * TPR * 8), t, TPR);  // pass 1's first batch
    if constexpr (OP == kAddRms) prefetch_l2(as<XT>(a.R) + off, min(D, UN * TPR * 8), t, TPR);
    pdl_enter();

    auto load = [&](int c0, float2 (&x)[UN][4], auto hint, bool keep_s) {
        constexpr int H = decltype(hint)::value;
#pragma unroll
        for (int u = 0; u < UN; ++u) {
            const int c = c0 + u * TPR;
            const bool v = c * 8 < D;
            ld_chunk<XT, H>(as<XT>(a.X) + off + c * 8, v, x[u]);
            if constexpr (OP == kAddRms) {
                float2 r[4];
                ld_chunk<XT, H>(as<XT>(a.R) + off + c * 8, v, r);
#pragma unroll
                for (int p = 0; p < 4; ++p) x[u][p] = __fadd2_rn(x[u][p], r[p]);
                if (keep_s && v) st_chunk<XT>(as<XT>(a.S) + off + c * 8, x[u]);
            }
        }
    };

    // LayerNorm: this thread's count, sum and centred sum of squares of x - k
    float n = 0.f, s = 0.f, m2 = 0.f;
    float2 q2 = make_float2(0.f, 0.f);  // RMSNorm, fused op: the sum of squares (chunks past D are 0)
    const float k = (OP == kLayer) ? ld_elem(a.X, off, XT) : 0.f;
    const float2 nk = make_float2(-k, -k);
    for (int c0 = t; c0 * 8 < D; c0 += UN * TPR) {
        float2 x[UN][4];
        load(c0, x, std::integral_constant<int, kReadOnly>{}, true);
        if constexpr (OP == kLayer) {
            float2 b2 = make_float2(0.f, 0.f);
            int nv = 0;
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                if ((c0 + u * TPR) * 8 >= D) continue;
                nv += 8;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    x[u][p] = __fadd2_rn(x[u][p], nk);
                    b2 = __fadd2_rn(b2, x[u][p]);
                }
            }
            const float nb = (float)nv, bs = b2.x + b2.y, bm = bs / nb;  // nv >= 8: chunk c0 is in the row
            const float2 nbm = make_float2(-bm, -bm);
            float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < UN; ++u) {
                if ((c0 + u * TPR) * 8 >= D) continue;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 d = __fadd2_rn(x[u][p], nbm);
                    d2 = __ffma2_rn(d, d, d2);
                }
            }
            const float bm2 = d2.x + d2.y;
            if (n == 0.f) {
                m2 = bm2;
            } else {
                const float dl = bm - s / n;
                m2 += bm2 + dl * dl * (n * nb / (n + nb));
            }
            s += bs;
            n += nb;
        } else {
#pragma unroll
            for (int u = 0; u < UN; ++u)
#pragma unroll
                for (int p = 0; p < 4; ++p) q2 = __ffma2_rn(x[u][p], x[u][p], q2);
        }
    }
    float mu = 0.f, q[1];  // LayerNorm: mu = mean(x - k)
    if constexpr (OP == kLayer) {
        float v[1] = {s};
        row_sum<TPR, 1, 1>(v, red, 0, 0, wir, lane);
        mu = v[0] * inv_d;
        const float dev = n > 0.f ? s / n - mu : 0.f;
        q[0] = m2 + n * dev * dev;
    } else {
        q[0] = q2.x + q2.y;
    }
    row_sum<TPR, 1, 1>(q, red, 1, 0, wir, lane);
    const float rs = rsqrtf(q[0] * inv_d + a.eps);
    if (t == 0) {
        a.rstd[row] = rs;
        if constexpr (OP == kLayer) a.mean[row] = k + mu;
    }

    // While this CTA applies its row (L2 reads, DRAM writes), warm L2 with the row that a CTA
    // of the next wave will take, `ahead` rows on: one bulk prefetch per array, thread 0.
    // Only rows of at most kStreamAheadBytes for RMSNorm, half that (all arrays) for
    // LayerNorm, whose rows take longer, so that a prefetched row waits longer in L2, and for
    // the fused op, whose first pass also writes S: a wave of larger rows, next to the rows
    // still waiting for their second pass, does not stay in L2. Measured on GB300: RMSNorm
    // 4096 x 32768 forward 84.2 -> 81.2 us, 2048 x 65536 97.6 -> 92.9 us, LayerNorm 4096 x
    // 32768 105.0 -> 96.6 us, fused 4096 x 16384 81.3 -> 79.7 us; with larger rows, LayerNorm
    // 2048 x 65536 110.2 -> 121.4 us, fused 4096 x 32768 160.0 -> 177.2 us, LayerNorm 1024 x
    // 131072 122.7 -> 144.8 us. Rows are 16-byte aligned and D % 8 == 0 on this path.
    {
        constexpr int ARR = (OP == kAddRms) ? 2 : 1;
        constexpr int64_t LIMIT = (OP == kRms) ? kStreamAheadBytes : kStreamAheadBytes / 2;
        const int64_t bytes = (int64_t)D * (int64_t)sizeof(*as<XT>(a.X));
        const int64_t nxt = row + a.ahead;
        if (t == 0 && a.ahead > 0 && nxt < a.N && ARR * bytes <= LIMIT) {
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(as<XT>(a.X) + nxt * D),
                         "r"((unsigned)bytes) : "memory");
            if constexpr (OP == kAddRms)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(as<XT>(a.R) + nxt * D),
                             "r"((unsigned)bytes) : "memory");
        }
    }
    const float2 rs2 = make_float2(rs, rs), nmu = make_float2(-mu, -mu);
    for (int c0 = t; c0 * 8 < D; c0 += UN * TPR) {
        float2 x[UN][4];
        load(c0, x, std::integral_constant<int, kStream>{}, false);
#pragma unroll
        for (int u = 0; u < UN; ++u) {
            const int col = (c0 + u * TPR) * 8;
            if (col >= D) continue;
            float2 g[4], y[4];
            ld_param<WT>(as<WT>(a.gamma) + col, g);
            if constexpr (OP == kLayer) {
                float2 b[4];
                ld_param<WT>(as<WT>(a.beta) + col, b);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 d = __fadd2_rn(__fadd2_rn(x[u][p], nk), nmu);  // (x - k) - mu
                    y[p] = __ffma2_rn(__fmul2_rn(d, rs2), g[p], b[p]);
                }
            } else {
#pragma unroll
                for (int p = 0; p < 4; ++p) y[p] = __fmul2_rn(__fmul2_rn(x[u][p], rs2), g[p]);
            }
            st_chunk<XT>(as<XT>(a.Y) + off + col, y);
        }
    }
}

// ----------------------------------------------------------------- backward ---
// Scalar fallback for any alignment and any width; types chosen at run time (a.xdt,
// a.wdt, a.gdt). Persistent: grid = P CTAs of TPR*RPC threads; CTA b processes row
// slots b*RPC + j*G*RPC (G = gridDim.x), row group rg taking row slot + rg.
// Dynamic shared memory (RPC > 1): NV x D floats for the fixed-order combine. Compiled
// for one resident CTA per SM, so the run-time type selection costs registers, not spills.
template <int OP, int TPR, int RPC, int CH, bool HAS_DS, bool CLU = false>
__global__ void __launch_bounds__(TPR * RPC, 1)
norm_bwd_kernel(const BwdArgs a) {
    pdl_enter();
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad launch shape");
    static_assert(!CLU || RPC == 1, "a split row is one row group per CTA");
    constexpr int WPR = TPR / 32;
    constexpr int NV = (OP == kLayer) ? 2 : 1;
    __shared__ float red[2 * RPC * WPR * NV];
    __shared__ float xch[CLU ? 2 * NV : 1];
    extern __shared__ float comb[];

    const int tid = threadIdx.x;
    const int rg = tid / TPR, t = tid % TPR, wir = t / 32, lane = tid % 32;
    const int D = a.D;
    const float inv_d = 1.0f / (float)D;
    const Window<CLU> win(D, a.slice);
    // split rows: every CTA of a cluster runs the cluster's rows (same count, same order)
    const int64_t owner = win.owner(), owners = win.owners();

    float accg[CH];
    float accb[(OP == kLayer) ? CH : 1];
#pragma unroll
    for (int k = 0; k < CH; ++k) accg[k] = 0.f;
#pragma unroll
    for (int k = 0; k < ((OP == kLayer) ? CH : 1); ++k) accb[k] = 0.f;

    int buf = 0;
    for (int64_t base = owner * RPC; base < a.N; base += owners * RPC, buf ^= 1) {
        const int64_t row = base + rg;
        const bool ok = row < a.N;
        if (WPR == 1 && !ok) continue;  // single-warp row group: no CTA barrier inside
        const int64_t off = (ok ? row : 0) * (int64_t)D;
        const int lim = ok ? win.end : 0;
        const float r = ok ? a.rstd[row] : 0.f;
        const float mu = (OP == kLayer && ok) ? a.mean[row] : 0.f;

        // Short row slices stay in registers between the passes; longer ones are read
        // again in pass 2 through L1 (where pass 1 left them), which avoids spills.
        constexpr bool KEEP = CH <= 8;
        float xs[KEEP ? CH : 1], dys[KEEP ? CH : 1];
        if constexpr (KEEP) {
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const int col = win.beg + k * TPR + t;
                xs[k] = col < lim ? ld_elem_stream(a.X, off + col, a.xdt) : 0.f;
                dys[k] = col < lim ? ld_elem_stream(a.dY, off + col, a.gdt) : 0.f;
            }
        }

        // pass 1: sum_j g*xhat and, for LayerNorm, sum_j g
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = 0.f;
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = win.beg + k * TPR + t;
            const bool in = col < lim;
            const float gm = in ? ld_elem(a.gamma, col, a.wdt) : 0.f;
            float xv, dv;
            if constexpr (KEEP) {
                xv = xs[k];
                dv = dys[k];
            } else {
                xv = in ? ld_elem(a.X, off + col, a.xdt) : 0.f;
                dv = in ? ld_elem(a.dY, off + col, a.gdt) : 0.f;
            }
            const float xh = (xv - mu) * r;
            const float g = dv * gm;
            v[0] += g * xh;
            if constexpr (OP == kLayer) v[NV - 1] += g;
        }
        row_sum<TPR, RPC, NV>(v, red, buf, rg, wir, lane);
        if constexpr (CLU) cluster_sum<NV>(v, xch, buf, win.cn);
        const float c = v[0] * inv_d;
        const float am = (OP == kLayer) ? v[NV - 1] * inv_d : 0.f;
        if (!ok) continue;

        // pass 2: dX and the parameter-gradient sums
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = win.beg + k * TPR + t;
            if (col >= win.end) continue;
            const float gm = ld_elem(a.gamma, col, a.wdt);
            float xv, dv;
            if constexpr (KEEP) {
                xv = xs[k];
                dv = dys[k];
            } else {
                xv = ld_elem(a.X, off + col, a.xdt);
                dv = ld_elem(a.dY, off + col, a.gdt);
            }
            const float xh = (xv - mu) * r;
            const float g = dv * gm;
            float dx = r * ((g - am) - xh * c);
            if constexpr (HAS_DS) dx += ld_elem_stream(a.dS, off + col, a.gdt);
            accg[k] += dv * xh;
            if constexpr (OP == kLayer) accb[k] += dv;
            st_elem(a.dX, off + col, dx, a.xdt);
        }
    }

    // Combine this CTA's row groups in the fixed order rg = 0, 1, ..., RPC-1 and
    // write one partial row per CTA. Thread t owns the same columns in every group.
    if constexpr (CLU) cluster_arrive();  // done reading the other CTAs' slots
    float *pg = a.part_g + (size_t)owner * D;
    float *pb = (OP == kLayer) ? a.part_b + (size_t)owner * D : nullptr;
    if constexpr (RPC == 1) {
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int col = win.beg + k * TPR + t;
            if (col >= win.end) continue;
            pg[col] = accg[k];
            if constexpr (OP == kLayer) pb[col] = accb[k];
        }
        if constexpr (CLU) cluster_wait();  // no CTA leaves while another may read its slots
    } else {
        float *cg = comb;
        float *cb = comb + D;
        for (int j = 0; j < RPC; ++j) {
            if (rg == j) {
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const int col = k * TPR + t;
                    if (col >= D) continue;
                    const float sg = (j == 0) ? accg[k] : cg[col] + accg[k];
                    if (j == RPC - 1) pg[col] = sg; else cg[col] = sg;
                    if constexpr (OP == kLayer) {
                        const float sb = (j == 0) ? accb[k] : cb[col] + accb[k];
                        if (j == RPC - 1) pb[col] = sb; else cb[col] = sb;
                    }
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace mt
