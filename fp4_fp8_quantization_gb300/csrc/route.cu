// Routing of top-k expert choices to expert groups: the local part of the
// expert-parallel token dispatch ("Struct_ep_dispatch_mxfp4", execute:
// row_offsets, expert_ids and src_info among its outputs; with one rank the
// all-to-all exchange is the identity).  Group e is expert e (empty groups
// kept); a group's rows hold its choices i = t * top_k + k in increasing i.
//
// One cluster of 16 CTAs (8, the portable size, where 16 cannot be
// resident) of 32 warps and no memory besides the
// caller's outputs.  CTA c owns a contiguous chunk of the choices and warp
// w of it a contiguous segment of that chunk.  Pass 1 builds one histogram
// per warp in shared memory; each CTA turns them into per-warp prefixes and
// its chunk's counts; after a cluster barrier every CTA reads the other
// CTAs' counts through distributed shared memory, which gives the expert
// totals (row offsets) and the first row of its chunk in each group.  Pass
// 2 walks each segment in order, 32 choices at a time, and ranks equal
// experts within the warp (match.any): a stable order with no atomics on
// the positions.  The scattered 4-byte stores of src_info are spread over
// the cluster's SMs; the inverse map dst_info (the row of each choice) is
// written in choice order.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moeq {

namespace {

constexpr int kRouteCtasMax = 16;  // non-portable cluster size, when it fits
constexpr int kRouteCtasPortable = 8;
constexpr int kRouteWarps = 32;
constexpr int kRouteThreads = kRouteWarps * 32;
constexpr int kRouteU = 16;  // 32-choice batches whose loads a warp issues together

// Exclusive prefix sums of two values over the block; returns the block
// totals in *t0, *t1.  Every thread of the block calls it.
__device__ __forceinline__ void block_exclusive_scan2(uint32_t &v0, uint32_t &v1, uint32_t *t0,
                                                      uint32_t *t1, uint32_t (*wsum)[2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t a = v0, b = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, a, o);
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, b, o);
        if (lane >= o) {
            a += x;
            b += y;
        }
    }
    if (lane == 31) {
        wsum[warp][0] = a;
        wsum[warp][1] = b;
    }
    __syncthreads();
    uint32_t ba = 0, bb = 0, ta = 0, tb = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
        if (w < warp) {
            ba += wsum[w][0];
            bb += wsum[w][1];
        }
        ta += wsum[w][0];
        tb += wsum[w][1];
    }
    v0 = ba + a - v0;
    v1 = bb + b - v1;
    *t0 = ta;
    *t1 = tb;
    __syncthreads();
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    route_topk_kernel(const int32_t *__restrict__ ids, int64_t n, int E, uint32_t *row_offsets,
                      int32_t *expert_ids, int32_t *src_info, int32_t *dst_info,
                      uint32_t *scales_offsets, int slot_rows, uint32_t *err) {
    // [kRouteWarps][E] per-warp histograms, then [E] chunk counts (read by
    // the other CTAs), [E] expert totals, [E] this chunk's offset in each group
    extern __shared__ uint32_t hist[];
    __shared__ uint32_t wsum[kRouteWarps][2];
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const int nct = (int)cluster_nctarank();
    uint32_t *cnt = hist + kRouteWarps * E;
    uint32_t *tot = cnt + E;
    uint32_t *before_chunk = tot + E;
    for (int i = threadIdx.x; i < (kRouteWarps + 1) * E; i += kRouteThreads) hist[i] = 0u;
    __syncthreads();

    // pass 1: per-warp histograms over contiguous segments of this chunk
    const int64_t per_cta = (n + nct - 1) / nct;
    const int64_t c0 = min(n, (int64_t)rank * per_cta), c1 = min(n, c0 + per_cta);
    const int64_t per = (c1 - c0 + kRouteWarps - 1) / kRouteWarps;
    const int64_t s0 = min(c1, c0 + (int64_t)warp * per), s1 = min(c1, s0 + per);
    uint32_t *h = hist + warp * E;
    bool bad = false;
    for (int64_t b = s0; b < s1; b += 32 * kRouteU) {
        int v[kRouteU];
#pragma unroll
        for (int u = 0; u < kRouteU; ++u) {
            const int64_t i = b + u * 32 + lane;
            v[u] = i < s1 ? __ldg(ids + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < kRouteU; ++u) {
            if (b + u * 32 + lane >= s1) continue;
            if (v[u] >= 0 && v[u] < E)
                atomicAdd(h + v[u], 1u);
            else
                bad = true;
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_error(err, MOEQ_DEVERR_BAD_EXPERT);
    __syncthreads();

    // per expert: segment counts -> exclusive prefix over the warps; chunk count
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
        uint32_t run = 0;
        for (int w = 0; w < kRouteWarps; ++w) {
            const uint32_t c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
        cnt[e] = run;
    }
    // every CTA's chunk counts are final and visible cluster-wide
    cluster_sync();

    // expert totals and this chunk's offset within each group, from the
    // counts of all CTAs (distributed shared memory); each thread takes a
    // contiguous run of experts
    const int chunk = (E + kRouteThreads - 1) / kRouteThreads;
    const int e0 = min(E, threadIdx.x * chunk), e1 = min(E, e0 + chunk);
    const uint32_t cnt_addr = smem_u32(cnt);
    uint32_t rows = 0, pad = 0;
    for (int e = e0; e < e1; ++e) {
        uint32_t t = 0, before = 0;
        for (int c = 0; c < nct; ++c) {
            const uint32_t v = ld_cluster_u32(mapa_shared(cnt_addr + 4u * e, (uint32_t)c));
            if (c < (int)rank) before += v;
            t += v;
        }
        tot[e] = t;
        before_chunk[e] = before;
        rows += t;
        pad += (t + 127u) & ~127u;
    }
    // no CTA leaves or rewrites its counts while another may still read them
    cluster_sync();

    // prefix over experts: row offsets and padded scale offsets
    uint32_t rows_total, pad_total;
    block_exclusive_scan2(rows, pad, &rows_total, &pad_total, wsum);
    for (int e = e0; e < e1; ++e) {
        if (rank == 0 && store_ok(e < E, err)) {
            row_offsets[e] = rows;
            expert_ids[e] = e;
            if (scales_offsets)
                scales_offsets[e] = slot_rows > 0 ? (uint32_t)e * (uint32_t)slot_rows : pad;
        }
        const uint32_t first = rows + before_chunk[e];  // this chunk's first row in group e
        for (int w = 0; w < kRouteWarps; ++w) hist[w * E + e] += first;
        rows += tot[e];
        pad += (tot[e] + 127u) & ~127u;
    }
    if (rank == 0 && threadIdx.x == 0) {
        row_offsets[E] = rows_total;
        if (scales_offsets)
            scales_offsets[E] = slot_rows > 0 ? (uint32_t)E * (uint32_t)slot_rows : pad_total;
    }
    __syncthreads();

    // pass 2: in-order scatter of each segment, 32 choices at a time (the
    // loads of kRouteU batches in flight together)
    const uint32_t lt = (1u << lane) - 1u;
    for (int64_t b = s0; b < s1; b += 32 * kRouteU) {
        int v[kRouteU];
#pragma unroll
        for (int u = 0; u < kRouteU; ++u) {
            const int64_t i = b + u * 32 + lane;
            v[u] = i < s1 ? __ldg(ids + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < kRouteU; ++u) {
            const int64_t i = b + u * 32 + lane;
            const bool ok = v[u] >= 0 && v[u] < E;
            const int e = ok ? v[u] : -1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
            uint32_t pos = 0;
            if (ok) pos = h[e] + __popc(peers & lt);
            __syncwarp();
            if (ok && (peers & lt) == 0) h[e] += __popc(peers);  // the group's lowest lane
            __syncwarp();
            if (ok && store_ok(pos < rows_total, err)) src_info[pos] = (int32_t)i;
            if (dst_info && i < s1) dst_info[i] = ok ? (int32_t)pos : -1;
        }
    }
}

}  // namespace

size_t route_smem_bytes(int num_experts) {
    return (size_t)(kRouteWarps + 3) * (size_t)num_experts * sizeof(uint32_t);
}

cudaError_t launch_route_topk(const int32_t *topk_ids, int64_t num_choices, int num_experts,
                              uint32_t *row_offsets, int32_t *expert_ids, int32_t *src_info,
                              int32_t *dst_info, uint32_t *scales_offsets, int slot_rows,
                              uint32_t *err, cudaStream_t s) {
    const size_t smem = route_smem_bytes(num_experts);
    // per device, the largest dynamic shared memory set so far and the
    // cluster size for the last shared-memory size queried; the set-up runs
    // under the library's launch lock (concurrent host threads)
    static size_t smem_set[kMaxDevices] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::unique_lock<std::mutex> lock(launch_setup_mutex());
    if (smem > 48 * 1024 && smem > smem_set[dev]) {
        e = cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        smem_set[dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = kPdl;
    cfg.blockDim = dim3(kRouteThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    // per device and shared-memory size: the cluster size that can be
    // resident (16 when the non-portable size fits, else 8)
    static int ctas_for[kMaxDevices] = {0};
    static size_t ctas_smem[kMaxDevices] = {0};
    if (!ctas_for[dev] || ctas_smem[dev] != smem) {
        int ctas = kRouteCtasPortable;
        if (cudaFuncSetAttribute(route_topk_kernel,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
            attr[0].val.clusterDim.x = kRouteCtasMax;
            cfg.gridDim = dim3(kRouteCtasMax, 1, 1);
            cfg.numAttrs = 1;
            int active = 0;
            if (cudaOccupancyMaxActiveClusters(&active, route_topk_kernel, &cfg) == cudaSuccess &&
                active >= 1)
                ctas = kRouteCtasMax;
        }
        cudaGetLastError();  // a refused query is not a launch error
        ctas_for[dev] = ctas;
        ctas_smem[dev] = smem;
    }
    const int ctas = ctas_for[dev];
    lock.unlock();
    attr[0].val.clusterDim.x = ctas;
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, route_topk_kernel, topk_ids, num_choices, num_experts,
                              row_offsets, expert_ids, src_info, dst_info, scales_offsets,
                              slot_rows, err);
}

}  // namespace moeq
