// Grouped activation quantizer (NVFP4 / MXFP8 / MXFP4), per-expert amax ->
// NVFP4 tensor scale, chained SwiGLU + NVFP4 requantization, padded scale
// offsets.  All are streaming (HBM-bound) kernels: one warp per logical
// (padded) scale row, 16-byte coalesced loads, block amax by warp shuffles,
// packed codes written as 4- or 8-byte coalesced stores, and block scales
// written one 4-byte word (four consecutive blocks of a row) at a time into
// the tiled 128x4 scale layout.
//
// Pages: "grouped_quantize_dynamic_scaled_fp4_async_kernel" (each block finds
// its expert by binary search on row_offsets / scales_offsets, then
// quantizes that expert's BF16 rows); "max.nn.moe.NvMxf4f8Strategy"
// (grouped_quantize: per-expert quantization with padded scales;
// fused_silu_quantize).
#include "common.cuh"
#include "launch.h"

namespace moeq {

namespace {

// Quantizer launch shape: warps per CTA, 32-byte loads in flight per lane,
// minimum resident CTAs per SM (which caps the registers).  CTAs of 4 warps,
// 4 loads per lane, at most 64 registers (8 CTAs per SM): against 8-warp
// CTAs with 62-72 registers, 9 % faster on 8192 x 4096 and 12 % on
// 131072 x 4096 rows (same box, back-to-back calls).
#ifndef MOEQ_Q_WARPS
#define MOEQ_Q_WARPS 4
#endif
#ifndef MOEQ_QUANT_U
#define MOEQ_QUANT_U 4
#endif
// NVFP4 rows: a rolling window of 32-byte loads per lane (the load of step
// s + W is issued as soon as step s is consumed).  3 in flight: 17.8 us on
// 8192 x 4096 rows against 18.4 us with 4 (same box, back-to-back calls).
#ifndef MOEQ_QUANT_W_NVFP4
#define MOEQ_QUANT_W_NVFP4 3
#endif
#ifndef MOEQ_Q_MINB
#define MOEQ_Q_MINB 8
#endif
constexpr int kQWarps = MOEQ_Q_WARPS;
// amax pass: warps per CTA on large inputs (>= 65536 rows) and on smaller
// ones (8192 x 4096: 14.3 us with 4-warp CTAs against 15.1 with 8; 131072 x
// 4096: 154 us with 8 against 164 with 4), rows per warp on large inputs
// (2 is 2 % faster than 4 on 131072 x 4096), min CTAs per SM
#ifndef MOEQ_A_WARPS
#define MOEQ_A_WARPS 8
#endif
#ifndef MOEQ_A_WARPS_SMALL
#define MOEQ_A_WARPS_SMALL 4
#endif
#ifndef MOEQ_A_RPW
#define MOEQ_A_RPW 2
#endif
#ifndef MOEQ_A_MINB
#define MOEQ_A_MINB 3  // at most 85 registers: 0.161 vs 0.173 ms unbounded (106 registers)
#endif
// chained SwiGLU (NVFP4 and MX outputs): persistent CTAs of kSWarps warps,
// MOEQ_SN_MINB per SM (each with its SiLU table), MOEQ_SN_RPW consecutive
// scale rows per warp and turn.  NVFP4 on 131072 x 3072: 0.186 ms with 16
// warps and 4 rows (0.189 / 0.197 ms with 2 / 8 rows; 32-warp CTAs 0.193
// ms); the same layout without the table and persistence 0.234 ms.
#ifndef MOEQ_S_WARPS
#define MOEQ_S_WARPS 16
#endif
constexpr int kSWarps = MOEQ_S_WARPS;
#ifndef MOEQ_SN_RPW
#define MOEQ_SN_RPW 4
#endif
#ifndef MOEQ_SN_MINB
#define MOEQ_SN_MINB 2
#endif

// The group description, read either from a per-CTA shared-memory copy
// (up to kTableCap groups: one coalesced round trip per CTA instead of a
// chain of dependent global loads per warp) or from global memory.
constexpr int kTableCap = 512;
struct GroupTable {
    uint32_t ro[kTableCap + 1];
    uint32_t so[kTableCap + 1];
    int32_t eid[kTableCap];
    float scale[kTableCap];  // per-group copy of the expert's fp32 scale
};

struct GroupView {
    const uint32_t *ro, *so;
    const int32_t *eid;
    const float *scale_g;  // per group (shared copy) or null
    const float *scale_e;  // per expert (global), used when scale_g is null
    int G, E;
    int64_t total_rows, scale_rows_total;
    __device__ __forceinline__ float scale(int g) const {
        return scale_g ? scale_g[g] : __ldg(scale_e + eid[g]);
    }
};

// Every thread of the CTA must call this (it synchronises the CTA).
__device__ __forceinline__ GroupView load_groups(const GroupArgs &g, const float *scale_e,
                                                 GroupTable &t) {
    GroupView v{g.row_offsets, g.scales_offsets, g.expert_ids, nullptr, scale_e,
                g.num_groups, g.num_experts, g.total_rows, g.scale_rows_total};
    if (g.num_groups <= kTableCap) {
        for (int i = threadIdx.x; i <= g.num_groups; i += blockDim.x) {
            t.ro[i] = __ldg(g.row_offsets + i);
            if (g.scales_offsets) t.so[i] = __ldg(g.scales_offsets + i);
            if (i < g.num_groups) {
                const int e = __ldg(g.expert_ids + i);
                t.eid[i] = e;
                t.scale[i] = (scale_e && e >= 0 && e < g.num_experts) ? __ldg(scale_e + e) : 1.0f;
            }
        }
        __syncthreads();
        v.ro = t.ro;
        v.so = g.scales_offsets ? t.so : nullptr;
        v.eid = t.eid;
        v.scale_g = t.scale;
    }
    return v;
}

// Largest g in [0, G) with offs[g] <= x (offs[0] <= x); plain loads, so the
// table may live in shared or global memory.
__device__ __forceinline__ int find_group(const uint32_t *offs, int G, uint32_t x) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offs[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

// Checks one group's offsets / expert id; returns true if it can be used.
__device__ __forceinline__ bool group_ok(const GroupView &g, int gi, uint32_t *err,
                                         bool need_scales) {
    const uint32_t r0 = g.ro[gi], r1 = g.ro[gi + 1];
    const int e = g.eid[gi];
    if (r1 < r0 || (int64_t)r1 > g.total_rows) {
        set_error(err, MOEQ_DEVERR_BAD_OFFSETS);
        return false;
    }
    if (e < 0 || e >= g.E) {
        set_error(err, MOEQ_DEVERR_BAD_EXPERT);
        return false;
    }
    if (need_scales) {
        const uint32_t s0 = g.so[gi], s1 = g.so[gi + 1];
        const uint32_t need = (r1 - r0 + 127u) & ~127u;
        if ((s0 & 127u) || s1 < s0 || s1 - s0 < need || (int64_t)s1 > g.scale_rows_total) {
            set_error(err, MOEQ_DEVERR_SCALE_ROWS);
            return false;
        }
    }
    return true;
}

// Maps logical scale row p to its group: returns g, or -1 when p lies in no
// group's scale range (or the group is invalid).
__device__ __forceinline__ int scale_row_group(const GroupView &g, uint32_t p, uint32_t *err) {
    const int G = g.G;
    if (p < g.so[0] || p >= g.so[G]) return -1;
    const int gi = find_group(g.so, G, p);
    if (p >= g.so[gi + 1]) return -1;
    return group_ok(g, gi, err, true) ? gi : -1;
}

// Sets the error bits of every invalid group without scale rows (one CTA
// calls it; the amax pass takes no scale offsets).
__device__ __forceinline__ void flag_bad_groups_rows(const GroupView &g, uint32_t *err) {
    for (int i = threadIdx.x; i < g.G; i += blockDim.x) group_ok(g, i, err, false);
}

__device__ __forceinline__ uint32_t bf16_abs_max8(const uint4 &v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = max(m, w[i] & 0x7FFFu);
        m = max(m, (w[i] >> 16) & 0x7FFFu);
    }
    return m;
}

// floor(log2(v)) of a non-zero non-negative bf16 given by its bits.
__device__ __forceinline__ int bf16_floor_log2(uint32_t b) {
    int ef = (int)((b >> 7) & 0xFFu);
    if (ef > 0) return ef - 127;
    return (31 - __clz((int)(b & 0x7Fu))) - 133;
}

// Gathers the byte `mine` of lanes base, base+step, base+2 step, base+3 step
// (base = this lane rounded down to 4*step) into one little-endian word.
__device__ __forceinline__ uint32_t gather4(uint32_t mine, int lane, int step) {
    int base = lane & ~(4 * step - 1);
    uint32_t b0 = __shfl_sync(0xFFFFFFFFu, mine, base);
    uint32_t b1 = __shfl_sync(0xFFFFFFFFu, mine, base + step);
    uint32_t b2 = __shfl_sync(0xFFFFFFFFu, mine, base + 2 * step);
    uint32_t b3 = __shfl_sync(0xFFFFFFFFu, mine, base + 3 * step);
    return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

__device__ __forceinline__ void zero_scale_row(uint8_t *scales, int64_t p, int64_t kv_atoms,
                                               int lane) {
    for (int64_t w = lane; w < kv_atoms; w += 32)
        *reinterpret_cast<uint32_t *>(scales + sf_word_offset(p, w, kv_atoms)) = 0u;
}

// --------------------------------------------------------------- amax pass

// Input row of quantized row `row`: row itself, or indices[row] / divisor
// when the rows are gathered; -1 (with the error bit set) when the index
// falls outside the input.
__device__ __forceinline__ int64_t source_row(const Gather &gt, int64_t row, uint32_t *err) {
    if (!gt.indices) return row;
    const int32_t v = __ldg(gt.indices + row);
    const int64_t s = v < 0 ? -1 : (int64_t)(v / gt.divisor);
    if (s < 0 || s >= gt.in_rows) {
        set_error(err, MOEQ_DEVERR_BAD_INDEX);
        return -1;
    }
    return s;
}

// First 8 x 16 bytes per lane of a row of n16 16-byte chunks (lane i:
// chunks i, i + 32, ..., i + 224); zeros past the row or without a row.
__device__ __forceinline__ void row_first_loads(const uint4 *src, int64_t n16, int lane,
                                                uint4 (&v)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int64_t c = lane + u * 32;
        v[u] = (src && c < n16) ? ld_stream(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// max |x| over one row of K bf16 as a bf16 bit pattern (NaN sorts above
// inf), the same value in every lane of the warp; v holds the row's first
// loads (row_first_loads).
__device__ __forceinline__ uint32_t row_abs_max(const uint4 *src, int64_t K, int lane,
                                                const uint4 (&v0)[8]) {
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) m = max(m, bf16_abs_max8(v0[u]));
    const int64_t n16 = K / 8;
    int64_t c = lane + 8 * 32;
    for (; c + 7 * 32 < n16; c += 8 * 32) {  // 8 independent loads in flight
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = ld_stream(src + c + u * 32);
#pragma unroll
        for (int u = 0; u < 8; ++u) m = max(m, bf16_abs_max8(v[u]));
    }
    for (; c < n16; c += 32) m = max(m, bf16_abs_max8(ld_stream(src + c)));
    return __reduce_max_sync(0xFFFFFFFFu, m);
}

// NW warps per CTA; the register bound follows from NW and MINB (large
// inputs: 85 registers for 3 resident 8-warp CTAs; small: 4-warp CTAs
// without a tighter bound than 3 per SM)
template <int NW, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB) amax_kernel(const uint16_t *__restrict__ in,
                                                   int64_t stride, int64_t K, GroupArgs g,
                                                   Gather gt,
                                                   uint32_t *__restrict__ amax_bits,
                                                   uint32_t *err, int rows_per_warp) {
    pdl_wait();
    pdl_trigger();
    __shared__ GroupTable table;
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t row_begin = warp_id * rows_per_warp;
    const int64_t n16 = K / 8;
    // the first row's first loads go out before the group table is read
    auto row_ptr = [&](int64_t row) -> const uint4 * {
        const int64_t srow = row < g.total_rows ? source_row(gt, row, nullptr) : -1;
        return srow >= 0 ? reinterpret_cast<const uint4 *>(in + srow * stride) : nullptr;
    };
    uint4 v[8];
    const uint4 *src = row_ptr(row_begin);
    row_first_loads(src, n16, lane, v);
    const GroupView gv = load_groups(g, nullptr, table);
    if (blockIdx.x == 0) flag_bad_groups_rows(gv, err);
    const int G = g.num_groups;
    const uint32_t first = gv.ro[0], last = gv.ro[G];
    int cur_e = -1;
    uint32_t cur_m = 0;
    for (int64_t i = 0; i < rows_per_warp; ++i) {
        const int64_t row = row_begin + i;
        if (row >= g.total_rows) break;
        if (i > 0) {
            src = row_ptr(row);
            row_first_loads(src, n16, lane, v);
        }
        if (row < first || row >= last) continue;
        const int gi = find_group(gv.ro, G, (uint32_t)row);
        if (row >= gv.ro[gi + 1] || row < gv.ro[gi] || !group_ok(gv, gi, nullptr, false)) continue;
        if (!src) {  // gathered index outside the input
            set_error(err, MOEQ_DEVERR_BAD_INDEX);
            continue;
        }
        const int e = gv.eid[gi];
        const uint32_t m = row_abs_max(src, K, lane, v);
        if (e != cur_e) {
            if (cur_e >= 0 && lane == 0 && cur_m && store_ok(cur_e < g.num_experts, err))
                atomicMax(amax_bits + cur_e, cur_m << 16);
            cur_e = e;
            cur_m = 0;
        }
        cur_m = max(cur_m, m);
    }
    if (cur_e >= 0 && lane == 0 && cur_m && store_ok(cur_e < g.num_experts, err))
        atomicMax(amax_bits + cur_e, cur_m << 16);
}

// Per-expert amax from tokens and their top-k expert ids: each token row is
// read once and its max |x| goes to every expert it chose (atomic max on the
// fp32 bits of the bf16 value), so the words equal amax_kernel's over the
// routed rows without reading a token once per choice.  An id outside
// [0, E) is skipped and sets MOEQ_DEVERR_BAD_EXPERT.
__global__ void __launch_bounds__(MOEQ_A_WARPS * 32, MOEQ_A_MINB)
    amax_topk_kernel(const uint16_t *__restrict__ in, int64_t stride, int64_t K,
                     int64_t num_tokens, const int32_t *__restrict__ topk, int top_k, int E,
                     uint32_t *__restrict__ amax_bits, uint32_t *err, int rows_per_warp) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n16 = K / 8;
    for (int64_t i = 0; i < rows_per_warp; ++i) {
        const int64_t t = warp_id * rows_per_warp + i;
        if (t >= num_tokens) break;
        const uint4 *src = reinterpret_cast<const uint4 *>(in + t * stride);
        uint4 v[8];
        row_first_loads(src, n16, lane, v);
        const uint32_t m = row_abs_max(src, K, lane, v);
        for (int j = lane; j < top_k; j += 32) {
            const int e = __ldg(topk + t * top_k + j);
            if (e < 0 || e >= E)
                set_error(err, MOEQ_DEVERR_BAD_EXPERT);
            else if (m && store_ok(e < E, err))
                atomicMax(amax_bits + e, m << 16);
        }
    }
}

// Zeroes the per-expert amax words before amax_kernel's atomics.
__global__ void zero_words_kernel(uint32_t *buf, int n) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) buf[i] = 0u;
}

// amax (fp32 bits of a bf16 value) -> s = amax / 2688, or 1 for amax == 0.
__global__ void amax_finalize_kernel(uint32_t *buf, int E) {
    pdl_wait();
    pdl_trigger();
    int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float amax = __uint_as_float(buf[e]);
    float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    reinterpret_cast<float *>(buf)[e] = s;
}

// ------------------------------------------------------------- quantizer

struct QuantParams {
    const uint16_t *in;
    int64_t stride, K;
    uint8_t *out;
    uint8_t *scales;
    const float *tensor_scale;
    GroupArgs g;
    Gather gt;
    uint32_t *err;
};

// 32 bytes (16 bf16) per lane, read once: one 256-bit load.
__device__ __forceinline__ void ld_stream32(const void *p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

// max |x| over 16 bf16 (bits), as a bf16 bit pattern.
__device__ __forceinline__ uint32_t bf16_abs_max16(const uint32_t (&w)[8]) {
    uint32_t m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[2 * i] & 0x7FFF7FFFu, b = w[2 * i + 1] & 0x7FFF7FFFu;
        asm("max.u16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(a), "r"(b));
    }
    asm("max.u16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[1]));
    asm("max.u16x2 %0, %1, %2;" : "=r"(m[2]) : "r"(m[2]), "r"(m[3]));
    asm("max.u16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[2]));
    return max(m[0] & 0xFFFFu, m[0] >> 16);
}

// The 32 bytes (16 bf16) of one 512-element step that a lane reads.
template <bool A32>
__device__ __forceinline__ void load_step(const uint8_t *a, uint32_t (&w)[8]) {
    if (A32) {  // row starts are 32-byte aligned: one 256-bit load
        ld_stream32(a, w);
    } else {
        const uint4 lo = ld_stream(a), hi = ld_stream(a + 16);
        w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
        w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
    }
}

// Entry c of the NVFP4 multiplier table: inv / value(c) for the E4M3 scale
// code c, 0 for the zero code (and the NaN code, never produced).
__device__ __forceinline__ float nvfp4_r_entry(uint32_t c, float inv) {
    return (c == 0 || c >= 0x7F) ? 0.0f : __fdiv_rn(inv, e4m3_pos_value(c));
}

// NVFP4 quantization of one row of K bf16 (one warp): lane i takes elements
// [16 i, 16 i + 16) of each 512-element step, a whole block.  Codes go to
// out_row, the E4M3 block scales to logical scale row prow.  The row's
// multiplier table r_tab[c] = inv / value(c) for every E4M3 code c (0 where
// the block scale is 0; the same IEEE division per entry as the block rule)
// is built while the row's first loads are in flight.
template <bool A32>
__device__ __forceinline__ void nvfp4_quantize_row(const uint8_t *src, uint8_t *out_row,
                                                   uint8_t *scales, int64_t prow, int64_t K,
                                                   float tscale, float *r_tab, int lane) {
    const int64_t kv_atoms = K / 64;
    const int nsteps = (int)((K + 511) / 512);
    const int lanes_last = (int)(K / 16 - (int64_t)(nsteps - 1) * 32);
    constexpr int U = MOEQ_QUANT_W_NVFP4;  // 32-byte loads in flight per lane
    // rolling window: step s is loaded into w[s % U]; once it is consumed,
    // the load of step s + U goes into the same registers
    uint32_t w[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[u][i] = 0u;
        if (u < nsteps && (u < nsteps - 1 || lane < lanes_last))
            load_step<A32>(src + (int64_t)u * 1024 + lane * 32, w[u]);
    }
    // the row's inverse tensor scale and multiplier table, while the first
    // loads are in flight
    const float inv = __fdiv_rn(1.0f, tscale);
#pragma unroll
    for (int j = 0; j < 4; ++j) r_tab[lane * 4 + j] = nvfp4_r_entry(lane * 4 + j, inv);
    __syncwarp();
    for (int s0 = 0; s0 < nsteps; s0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u;
            if (s >= nsteps) break;
            const bool active = s < nsteps - 1 || lane < lanes_last;
            const uint32_t mb = bf16_abs_max16(w[u]);
            const Nvfp4Scale sc0 = nvfp4_block_scale_code(bf16_bits_to_f32(mb), inv);
            const float r = r_tab[sc0.code];
            float x[8];
            uint32_t codes[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[2 * i] = bf16_bits_to_f32(w[u][4 * h + i] & 0xFFFFu);
                    x[2 * i + 1] = __uint_as_float(w[u][4 * h + i] & 0xFFFF0000u);
                }
                codes[h] = nvfp4_codes8(x, r);
            }
            const int sn = s + U;
#pragma unroll
            for (int i = 0; i < 8; ++i) w[u][i] = 0u;
            if (sn < nsteps && (sn < nsteps - 1 || lane < lanes_last))
                load_step<A32>(src + (int64_t)sn * 1024 + lane * 32, w[u]);
            const uint32_t word = gather4(sc0.code, lane, 1);
            if (!active) continue;
            reinterpret_cast<uint2 *>(out_row)[s * 32 + lane] = make_uint2(codes[0], codes[1]);
            if ((lane & 3) == 0)
                *reinterpret_cast<uint32_t *>(
                    scales + sf_word_offset(prow, s * 8 + (lane >> 2), kv_atoms)) = word;
        }
    }
}


// fmt: 0 NVFP4, 1 MXFP4, 2 MXFP8.  One warp per logical scale row; in each
// 512-element step lane i takes elements [16 i, 16 i + 16): a whole NVFP4
// block, or half of an MX block (lanes 2j, 2j+1 share block j).
template <int FMT, bool A32>
__global__ void __launch_bounds__(kQWarps * 32, MOEQ_Q_MINB) quantize_kernel(QuantParams p) {
    pdl_wait();
    pdl_trigger();
    __shared__ float r_table[kQWarps][128];
    __shared__ GroupTable table;
    // the group table without the tensor scales: a row's scale is read when
    // the row starts, so that its load overlaps the row's first loads
    // instead of adding a second round trip before the CTA barrier
    GroupView gv = load_groups(p.g, nullptr, table);
    if (FMT == 0) {
        gv.scale_g = nullptr;
        gv.scale_e = p.tensor_scale;
    }
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int64_t prow = (int64_t)blockIdx.x * kQWarps + wid;
    if (prow >= p.g.scale_rows_total) return;
    const int gi = scale_row_group(gv, (uint32_t)prow, p.err);
    if (gi < 0) return;
    constexpr int V = FMT == 0 ? 16 : 32;
    const int64_t kv_atoms = p.K / V / 4;
    const uint32_t r0 = gv.ro[gi];
    const uint32_t rg = gv.ro[gi + 1] - r0;
    const uint32_t local = (uint32_t)prow - gv.so[gi];
    if (local >= rg) {  // padding row of this group (up to the next multiple of 128)
        if (local < ((rg + 127u) & ~127u) && store_ok(prow < p.g.scale_rows_total, p.err))
            zero_scale_row(p.scales, prow, kv_atoms, lane);
        return;
    }
    const int64_t row = (int64_t)r0 + local;
    if (!store_ok(row < p.g.total_rows && prow < p.g.scale_rows_total, p.err)) return;
    const int64_t srow = source_row(p.gt, row, p.err);  // gathered input row
    if (srow < 0) return;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(p.in + srow * p.stride);
    if (FMT == 0) {
        // r depends only on the block's E4M3 scale code: tabulated per row
        nvfp4_quantize_row<A32>(src, p.out + row * (p.K / 2), p.scales, prow, p.K, gv.scale(gi),
                                r_table[wid], lane);
        return;
    }
    const int nsteps = (int)((p.K + 511) / 512);
    const int lanes_last = (int)(p.K / 16 - (int64_t)(nsteps - 1) * 32);
    constexpr int U = MOEQ_QUANT_U;  // 32-byte loads in flight per lane
    for (int s0 = 0; s0 < nsteps; s0 += U) {
        uint32_t w[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[u][i] = 0u;
            const int s = s0 + u;
            if (s < nsteps && (s < nsteps - 1 || lane < lanes_last))
                load_step<A32>(src + (int64_t)s * 1024 + lane * 32, w[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u;
            if (s >= nsteps) break;
            const bool active = s < nsteps - 1 || lane < lanes_last;
            uint32_t mb = bf16_abs_max16(w[u]);
            {  // MX block: lanes 2j and 2j+1
                mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
                constexpr int emax = FMT == 2 ? 8 : 2;
                uint32_t code = 0;
                float f = 0.0f;
                if (mb != 0) {
                    int cs = bf16_floor_log2(mb) - emax + 127;
                    cs = min(max(cs, 0), 254);
                    code = (uint32_t)cs;
                    f = __uint_as_float((uint32_t)(254 - cs) << 23);  // 2^(127-c)
                }
                uint32_t o[4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float y[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        y[2 * i] = __fmul_rn(bf16_bits_to_f32(w[u][4 * h + i] & 0xFFFFu), f);
                        y[2 * i + 1] = __fmul_rn(__uint_as_float(w[u][4 * h + i] & 0xFFFF0000u), f);
                    }
                    if (FMT == 2) {
                        o[2 * h] = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
                        o[2 * h + 1] = e4m3x2(y[4], y[5]) | (e4m3x2(y[6], y[7]) << 16);
                    } else {
                        o[h] = e2m1x8(y);
                    }
                }
                if (mb == 0) o[0] = o[1] = o[2] = o[3] = 0u;  // all-zero block: +0 codes
                const uint32_t word = gather4(code, lane, 2);
                if (!active) continue;
                if (FMT == 2)
                    st_global_v4(p.out + row * p.K + (int64_t)s * 512 + lane * 16, o[0], o[1], o[2],
                                 o[3]);
                else
                    reinterpret_cast<uint2 *>(p.out + row * (p.K / 2))[s * 32 + lane] =
                        make_uint2(o[0], o[1]);
                if ((lane & 7) == 0)
                    *reinterpret_cast<uint32_t *>(
                        p.scales + sf_word_offset(prow, s * 4 + (lane >> 3), kv_atoms)) = word;
            }
        }
    }
}

// ------------------------------------------- token-major quantization

// Token-major form of the gathered quantizer for routed tokens: one warp per
// token reads the token's row once and writes every routed copy of it
// (routed row dst[t * top_k + j] of expert topk[t * top_k + j]), with the
// same per-row arithmetic as quantize_kernel on the gathered rows, so the
// bytes are those of moeq_grouped_quantize_gather with indices = src_info
// and divisor = top_k.  MX formats: one quantization per block, stored
// top_k times.  NVFP4: the block amax and the loads are shared, the scale
// code and the element codes use each expert's tensor scale (per-choice
// multiplier tables in shared memory).  Padding scale rows are zeroed by
// zero_padding_scale_rows_kernel.
constexpr int kTopkMax = 8;

struct TopkQuantParams {
    const uint16_t *in;
    int64_t stride, K, num_tokens;
    const int32_t *topk, *dst;  // [num_tokens * top_k]
    int top_k, E;
    const uint32_t *ro, *so;    // [E + 1]
    const float *tensor_scale;  // NVFP4
    int64_t total_rows, scale_rows_total;
    uint8_t *out, *scales;
    uint32_t *err;
};

// Routed row and logical scale row of choice (t, j), -1 when the choice is
// dropped or its group cannot hold its scale rows (then flagged).
__device__ __forceinline__ void topk_choice(const TopkQuantParams &p, int64_t i, int64_t &row,
                                            int64_t &prow, int &e) {
    row = prow = -1;
    e = __ldg(p.topk + i);
    const int pos = __ldg(p.dst + i);
    if (e < 0 || e >= p.E || pos < 0) return;  // dropped by the router (already flagged)
    const uint32_t r0 = __ldg(p.ro + e), r1 = __ldg(p.ro + e + 1);
    const uint32_t s0 = __ldg(p.so + e), s1 = __ldg(p.so + e + 1);
    if (r1 < r0 || (int64_t)r1 > p.total_rows || (uint32_t)pos < r0 || (uint32_t)pos >= r1) {
        set_error(p.err, MOEQ_DEVERR_BAD_OFFSETS);
        return;
    }
    const uint32_t need = (r1 - r0 + 127u) & ~127u;
    if ((s0 & 127u) || s1 < s0 || s1 - s0 < need || (int64_t)s1 > p.scale_rows_total) {
        set_error(p.err, MOEQ_DEVERR_SCALE_ROWS);
        return;
    }
    row = pos;
    prow = (int64_t)s0 + (pos - r0);
}

template <int FMT, bool A32>
__global__ void __launch_bounds__(kQWarps * 32, MOEQ_Q_MINB)
    quantize_topk_kernel(TopkQuantParams p) {
    pdl_wait();
    pdl_trigger();
    __shared__ float r_table[FMT == 0 ? kQWarps : 1][FMT == 0 ? kTopkMax : 1][128];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * kQWarps + wid;
    if (t >= p.num_tokens) return;
    // lane j < top_k holds choice j's routed row, scale row and inverse scale
    int64_t my_row = -1, my_prow = -1;
    float my_inv = 0.0f;
    if (lane < p.top_k) {
        int e;
        topk_choice(p, t * p.top_k + lane, my_row, my_prow, e);
        if (FMT == 0 && my_row >= 0) my_inv = __fdiv_rn(1.0f, __ldg(p.tensor_scale + e));
    }
    if (FMT == 0) {
        for (int j = 0; j < p.top_k; ++j) {
            const float inv = __shfl_sync(0xFFFFFFFFu, my_inv, j);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                r_table[wid][j][lane * 4 + c] = nvfp4_r_entry(lane * 4 + c, inv);
        }
        __syncwarp();
    }
    constexpr int V = FMT == 0 ? 16 : 32;
    const int64_t kv_atoms = p.K / V / 4;
    const int64_t ob = FMT == 2 ? p.K : p.K / 2;  // output bytes per row
    const uint8_t *src = reinterpret_cast<const uint8_t *>(p.in + t * p.stride);
    const int nsteps = (int)((p.K + 511) / 512);
    const int lanes_last = (int)(p.K / 16 - (int64_t)(nsteps - 1) * 32);
    constexpr int U = 2;  // 32-byte loads in flight per lane
    for (int s0 = 0; s0 < nsteps; s0 += U) {
        uint32_t w[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[u][i] = 0u;
            const int s = s0 + u;
            if (s < nsteps && (s < nsteps - 1 || lane < lanes_last))
                load_step<A32>(src + (int64_t)s * 1024 + lane * 32, w[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u;
            if (s >= nsteps) break;
            const bool active = s < nsteps - 1 || lane < lanes_last;
            uint32_t mb = bf16_abs_max16(w[u]);
            if (FMT == 0) {
                float x[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[h][2 * i] = bf16_bits_to_f32(w[u][4 * h + i] & 0xFFFFu);
                        x[h][2 * i + 1] = __uint_as_float(w[u][4 * h + i] & 0xFFFF0000u);
                    }
                }
                const float mf = bf16_bits_to_f32(mb);
                for (int j = 0; j < p.top_k; ++j) {
                    const int64_t row = __shfl_sync(0xFFFFFFFFu, my_row, j);
                    const int64_t prow = __shfl_sync(0xFFFFFFFFu, my_prow, j);
                    const float inv = __shfl_sync(0xFFFFFFFFu, my_inv, j);
                    if (row < 0) continue;  // the same for every lane
                    const uint32_t code = nvfp4_block_scale_code(mf, inv).code;
                    const float r = r_table[wid][j][code];
                    const uint32_t c0 = nvfp4_codes8(x[0], r), c1 = nvfp4_codes8(x[1], r);
                    const uint32_t word = gather4(code, lane, 1);
                    if (!active) continue;
                    if (!store_ok(row < p.total_rows && prow < p.scale_rows_total, p.err))
                        continue;
                    reinterpret_cast<uint2 *>(p.out + row * ob)[s * 32 + lane] = make_uint2(c0, c1);
                    if ((lane & 3) == 0)
                        *reinterpret_cast<uint32_t *>(
                            p.scales + sf_word_offset(prow, s * 8 + (lane >> 2), kv_atoms)) = word;
                }
            } else {
                mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));  // lanes 2j, 2j+1
                constexpr int emax = FMT == 2 ? 8 : 2;
                uint32_t code = 0;
                float f = 0.0f;
                if (mb != 0) {
                    int cs = bf16_floor_log2(mb) - emax + 127;
                    cs = min(max(cs, 0), 254);
                    code = (uint32_t)cs;
                    f = __uint_as_float((uint32_t)(254 - cs) << 23);  // 2^(127-c)
                }
                uint32_t o[4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float y[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        y[2 * i] = __fmul_rn(bf16_bits_to_f32(w[u][4 * h + i] & 0xFFFFu), f);
                        y[2 * i + 1] = __fmul_rn(__uint_as_float(w[u][4 * h + i] & 0xFFFF0000u), f);
                    }
                    if (FMT == 2) {
                        o[2 * h] = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
                        o[2 * h + 1] = e4m3x2(y[4], y[5]) | (e4m3x2(y[6], y[7]) << 16);
                    } else {
                        o[h] = e2m1x8(y);
                    }
                }
                if (mb == 0) o[0] = o[1] = o[2] = o[3] = 0u;  // all-zero block: +0 codes
                const uint32_t word = gather4(code, lane, 2);
                for (int j = 0; j < p.top_k; ++j) {
                    const int64_t row = __shfl_sync(0xFFFFFFFFu, my_row, j);
                    const int64_t prow = __shfl_sync(0xFFFFFFFFu, my_prow, j);
                    if (row < 0 || !active) continue;
                    if (!store_ok(row < p.total_rows && prow < p.scale_rows_total, p.err))
                        continue;
                    if (FMT == 2)
                        st_global_v4(p.out + row * ob + (int64_t)s * 512 + lane * 16, o[0], o[1],
                                     o[2], o[3]);
                    else
                        reinterpret_cast<uint2 *>(p.out + row * ob)[s * 32 + lane] =
                            make_uint2(o[0], o[1]);
                    if ((lane & 7) == 0)
                        *reinterpret_cast<uint32_t *>(
                            p.scales + sf_word_offset(prow, s * 4 + (lane >> 3), kv_atoms)) = word;
                }
            }
        }
    }
}

// Zero scale words of every group's padding rows, [so[e] + r_e,
// so[e] + ceil128(r_e)), for groups whose scale rows fit (as the grouped
// quantizer writes them); one CTA per group.
__global__ void zero_padding_scale_rows_kernel(const uint32_t *ro, const uint32_t *so, int E,
                                               int64_t total_rows, int64_t scale_rows_total,
                                               int64_t kv_atoms, uint8_t *scales, uint32_t *err) {
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.x;
    if (e >= E) return;
    const uint32_t r0 = __ldg(ro + e), r1 = __ldg(ro + e + 1);
    const uint32_t s0 = __ldg(so + e), s1 = __ldg(so + e + 1);
    if (r1 < r0 || (int64_t)r1 > total_rows) return;
    const uint32_t rg = r1 - r0, need = (rg + 127u) & ~127u;
    if ((s0 & 127u) || s1 < s0 || s1 - s0 < need || (int64_t)s1 > scale_rows_total) return;
    const int64_t nwords = (int64_t)(need - rg) * kv_atoms;
    for (int64_t k = threadIdx.x; k < nwords; k += blockDim.x) {
        const int64_t prow = (int64_t)s0 + rg + k / kv_atoms;
        if (store_ok(prow < scale_rows_total, err))
            *reinterpret_cast<uint32_t *>(scales + sf_word_offset(prow, k % kv_atoms, kv_atoms)) = 0u;
    }
}

// --------------------------------------------- chained SwiGLU + NVFP4

struct SwigluParams {
    const uint16_t *y;   // [T, 2I] bf16
    int64_t I;
    uint8_t *out;        // NVFP4 / MXFP4 [T, I/2], MXFP8 [T, I]
    uint8_t *scales;
    const float *out_tensor_scale;  // NVFP4 only
    GroupArgs g;
    uint32_t *err;
};

// SwiGLU + NVFP4 requant of one row of y (one warp).  In each 512-h step
// lane i takes the (gate, up) pairs of h [16 i, 16 i + 16), one whole NVFP4
// block: 64 bytes of y, read as two 32-byte loads (four 16-byte loads when
// y is not 32-byte aligned).  The loads of step s + 1 are issued as soon as
// the pairs of step s are turned into h, so they are in flight while step s
// is quantized.  r_tab is the row group's multiplier table (entry c = inv /
// value(c), 0 where value(c) is 0: the division of the block rule, once per
// code).  Codes go to out_row (8 bytes per lane and step), the E4M3 block
// scales to logical scale row prow (one 4-byte word per 4 lanes).
template <bool A32>
__device__ __forceinline__ void swiglu_nvfp4_row(const uint8_t *src, uint8_t *out_row,
                                                 uint8_t *scales, int64_t prow, int nh,
                                                 int64_t kv_atoms, float inv,
                                                 const float *r_tab, const float *silu_tab,
                                                 int lane) {
    const int nsteps = (nh + 511) >> 9;
    const int lanes_last = (nh - ((nsteps - 1) << 9)) >> 4;  // nh is a multiple of 64
    auto load = [&](int s, uint32_t (&d)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) d[i] = 0u;
        if (s >= nsteps || (s == nsteps - 1 && lane >= lanes_last)) return;
        const uint8_t *a = src + ((int64_t)s << 11) + lane * 64;
        if (A32) {
            ld_stream32(a, *reinterpret_cast<uint32_t(*)[8]>(&d[0]));
            ld_stream32(a + 32, *reinterpret_cast<uint32_t(*)[8]>(&d[8]));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = ld_stream(a + 16 * k);
                d[4 * k] = v.x;
                d[4 * k + 1] = v.y;
                d[4 * k + 2] = v.z;
                d[4 * k + 3] = v.w;
            }
        }
    };
    uint32_t w[16];
    load(0, w);
    // the scale word of blocks [4 kb, 4 kb + 4) of this row is at sf0 + 512 kb
    const int64_t sf0 = sf_word_offset(prow, 0, kv_atoms);
    for (int s = 0; s < nsteps; ++s) {
        const bool active = s < nsteps - 1 || lane < lanes_last;
        float h[16];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {  // word i: gate_i in the low half, up_i in the high
            const F2 hh = swiglu2_tab(w[i], w[i + 1], silu_tab);
            h[i] = f2_lo(hh);
            h[i + 1] = f2_hi(hh);
        }
        load(s + 1, w);
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(h[i]));
        const uint32_t code = nvfp4_block_scale_code(m, inv).code;
        const float r = r_tab[code & 0x7Fu];
        float lo8[8], hi8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo8[i] = h[i];
            hi8[i] = h[8 + i];
        }
        const uint32_t c0 = nvfp4_codes8(lo8, r);
        const uint32_t c1 = nvfp4_codes8(hi8, r);
        // lanes 4j .. 4j+3 hold the scale bytes of one word
        uint32_t word = code << (8 * (lane & 3));
        word |= __shfl_xor_sync(0xFFFFFFFFu, word, 1);
        word |= __shfl_xor_sync(0xFFFFFFFFu, word, 2);
        if (!active) continue;
        reinterpret_cast<uint2 *>(out_row)[s * 32 + lane] = make_uint2(c0, c1);
        if ((lane & 3) == 0)
            *reinterpret_cast<uint32_t *>(scales + sf0 + (int64_t)(s * 8 + (lane >> 2)) * 512) =
                word;
    }
}

// Chained SwiGLU + NVFP4: persistent CTAs; each builds the SiLU table in
// dynamic shared memory, then each warp takes MOEQ_SN_RPW consecutive
// logical scale rows per turn, looking their group up (and building its
// multiplier table) only when a row leaves the group of the previous one.
__global__ void __launch_bounds__(kSWarps * 32, MOEQ_SN_MINB) swiglu_nvfp4_kernel(SwigluParams p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float silu_tab[];
    __shared__ float r_tables[kSWarps][128];
    __shared__ GroupTable table;
    build_silu_table(silu_tab);
    const GroupView gv = load_groups(p.g, p.out_tensor_scale, table);  // (CTA barrier)
    const int lane = threadIdx.x & 31;
    float *r_tab = r_tables[threadIdx.x >> 5];
    const int64_t kv_atoms = p.I / 64;
    const bool a32 = (reinterpret_cast<uintptr_t>(p.y) & 31) == 0;
    int gi = -1;
    uint32_t s0 = 0, s1 = 0, r0 = 0, rg = 0;
    float inv = 0.0f;
    const int64_t turn = (int64_t)gridDim.x * kSWarps * MOEQ_SN_RPW;
    for (int64_t prow0 = ((int64_t)blockIdx.x * kSWarps + (threadIdx.x >> 5)) * MOEQ_SN_RPW;
         prow0 < p.g.scale_rows_total; prow0 += turn)
    for (int k = 0; k < MOEQ_SN_RPW; ++k) {
        const int64_t prow = prow0 + k;  // warp-uniform
        if (prow >= p.g.scale_rows_total) break;
        if (gi < 0 || (uint32_t)prow < s0 || (uint32_t)prow >= s1) {
            gi = scale_row_group(gv, (uint32_t)prow, p.err);
            if (gi < 0) continue;
            s0 = gv.so[gi];
            s1 = gv.so[gi + 1];
            r0 = gv.ro[gi];
            rg = gv.ro[gi + 1] - r0;
            inv = __fdiv_rn(1.0f, gv.scale(gi));
            __syncwarp();  // every lane is done with the previous table
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t c = (uint32_t)(lane * 4 + j);
                const float v = e4m3_pos_value(c);
                r_tab[c] = v == 0.0f ? 0.0f : __fdiv_rn(inv, v);
            }
            __syncwarp();
        }
        const uint32_t local = (uint32_t)prow - s0;
        if (local >= rg) {  // padding row of the group
            if (local < ((rg + 127u) & ~127u) && store_ok(prow < p.g.scale_rows_total, p.err))
                zero_scale_row(p.scales, prow, kv_atoms, lane);
            continue;
        }
        const int64_t row = (int64_t)r0 + local;
        if (!store_ok(row < p.g.total_rows, p.err)) continue;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.y + row * 2 * p.I);
        uint8_t *out_row = p.out + row * (p.I / 2);
        if (a32)
            swiglu_nvfp4_row<true>(src, out_row, p.scales, prow, (int)p.I, kv_atoms, inv, r_tab,
                                   silu_tab, lane);
        else
            swiglu_nvfp4_row<false>(src, out_row, p.scales, prow, (int)p.I, kv_atoms, inv, r_tab,
                                    silu_tab, lane);
    }
}

// SwiGLU + MX requant of one row of y (one warp).  In each 512-h step lane
// i takes the (gate, up) pairs of h [16 i, 16 i + 16): an MX block of 32 h
// is held by lanes 2j, 2j + 1.  As in the NVFP4 row, the next step's loads
// are issued once the current pairs are turned into h.  OUT: 1 MXFP4 (8
// bytes per lane and step), 2 MXFP8 (16 bytes); the E8M0 scales go to
// logical scale row prow (one 4-byte word per 8 lanes).
template <int OUT, bool A32>
__device__ __forceinline__ void swiglu_mx_row(const uint8_t *src, uint8_t *out_row,
                                              uint8_t *scales, int64_t prow, int nh,
                                              int64_t kv_atoms, const float *silu_tab, int lane) {
    const int nsteps = (nh + 511) >> 9;
    const int lanes_last = (nh - ((nsteps - 1) << 9)) >> 4;  // nh is a multiple of 128
    auto load = [&](int s, uint32_t (&d)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) d[i] = 0u;
        if (s >= nsteps || (s == nsteps - 1 && lane >= lanes_last)) return;
        const uint8_t *a = src + ((int64_t)s << 11) + lane * 64;
        if (A32) {
            ld_stream32(a, *reinterpret_cast<uint32_t(*)[8]>(&d[0]));
            ld_stream32(a + 32, *reinterpret_cast<uint32_t(*)[8]>(&d[8]));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = ld_stream(a + 16 * k);
                d[4 * k] = v.x;
                d[4 * k + 1] = v.y;
                d[4 * k + 2] = v.z;
                d[4 * k + 3] = v.w;
            }
        }
    };
    uint32_t w[16];
    load(0, w);
    const int64_t sf0 = sf_word_offset(prow, 0, kv_atoms);
    for (int s = 0; s < nsteps; ++s) {
        const bool active = s < nsteps - 1 || lane < lanes_last;
        float h[16];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {  // word i: gate_i in the low half, up_i in the high
            const F2 hh = swiglu2_tab(w[i], w[i + 1], silu_tab);
            h[i] = f2_lo(hh);
            h[i + 1] = f2_hi(hh);
        }
        load(s + 1, w);
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(h[i]));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));  // the block's two lanes
        uint32_t code = 0;
        float f = 0.0f;
        if (m != 0.0f) {
            code = mx_scale_code_f32(m, OUT == 2 ? 8 : 2);
            f = mx_multiplier(code);
        }
        const F2 f2v = f2(f, f);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const F2 t = mul2(f2(h[i], h[i + 1]), f2v);
            h[i] = f2_lo(t);
            h[i + 1] = f2_hi(t);
        }
        // lanes 8j .. 8j+7 hold the scale bytes of one word (two lanes per byte)
        uint32_t word = code << (8 * ((lane >> 1) & 3));
        word |= __shfl_xor_sync(0xFFFFFFFFu, word, 2);
        word |= __shfl_xor_sync(0xFFFFFFFFu, word, 4);
        if (!active) continue;
        if (OUT == 2) {
            uint4 o;
            o.x = e4m3x2(h[0], h[1]) | (e4m3x2(h[2], h[3]) << 16);
            o.y = e4m3x2(h[4], h[5]) | (e4m3x2(h[6], h[7]) << 16);
            o.z = e4m3x2(h[8], h[9]) | (e4m3x2(h[10], h[11]) << 16);
            o.w = e4m3x2(h[12], h[13]) | (e4m3x2(h[14], h[15]) << 16);
            if (m == 0.0f) o = make_uint4(0u, 0u, 0u, 0u);  // all-zero block: +0 codes
            reinterpret_cast<uint4 *>(out_row)[s * 32 + lane] = o;
        } else {
            float lo8[8], hi8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lo8[i] = h[i];
                hi8[i] = h[8 + i];
            }
            uint2 o = make_uint2(e2m1x8(lo8), e2m1x8(hi8));
            if (m == 0.0f) o = make_uint2(0u, 0u);
            reinterpret_cast<uint2 *>(out_row)[s * 32 + lane] = o;
        }
        if ((lane & 7) == 0)
            *reinterpret_cast<uint32_t *>(scales + sf0 + (int64_t)(s * 4 + (lane >> 3)) * 512) =
                word;
    }
}

// Chained SwiGLU + MX requant (OUT: 1 MXFP4, 2 MXFP8): persistent CTAs
// with the SiLU table, MOEQ_SN_RPW consecutive logical scale rows per warp
// and turn, the group looked up only when a row leaves the previous one's.
template <int OUT>
__global__ void __launch_bounds__(kSWarps * 32, MOEQ_SN_MINB) swiglu_mx_kernel(SwigluParams p) {
    static_assert(OUT == 1 || OUT == 2, "MX output formats");
    pdl_wait();
    pdl_trigger();
    extern __shared__ float silu_tab[];
    __shared__ GroupTable table;
    build_silu_table(silu_tab);
    const GroupView gv = load_groups(p.g, nullptr, table);  // (CTA barrier)
    const int lane = threadIdx.x & 31;
    const int64_t kv_atoms = p.I / 128;
    const int64_t ob = OUT == 2 ? p.I : p.I / 2;  // output bytes per row
    const bool a32 = (reinterpret_cast<uintptr_t>(p.y) & 31) == 0;
    int gi = -1;
    uint32_t s0 = 0, s1 = 0, r0 = 0, rg = 0;
    const int64_t turn = (int64_t)gridDim.x * kSWarps * MOEQ_SN_RPW;
    for (int64_t prow0 = ((int64_t)blockIdx.x * kSWarps + (threadIdx.x >> 5)) * MOEQ_SN_RPW;
         prow0 < p.g.scale_rows_total; prow0 += turn)
    for (int k = 0; k < MOEQ_SN_RPW; ++k) {
        const int64_t prow = prow0 + k;  // warp-uniform
        if (prow >= p.g.scale_rows_total) break;
        if (gi < 0 || (uint32_t)prow < s0 || (uint32_t)prow >= s1) {
            gi = scale_row_group(gv, (uint32_t)prow, p.err);
            if (gi < 0) continue;
            s0 = gv.so[gi];
            s1 = gv.so[gi + 1];
            r0 = gv.ro[gi];
            rg = gv.ro[gi + 1] - r0;
        }
        const uint32_t local = (uint32_t)prow - s0;
        if (local >= rg) {  // padding row of the group
            if (local < ((rg + 127u) & ~127u) && store_ok(prow < p.g.scale_rows_total, p.err))
                zero_scale_row(p.scales, prow, kv_atoms, lane);
            continue;
        }
        const int64_t row = (int64_t)r0 + local;
        if (!store_ok(row < p.g.total_rows, p.err)) continue;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.y + row * 2 * p.I);
        uint8_t *out_row = p.out + row * ob;
        if (a32)
            swiglu_mx_row<OUT, true>(src, out_row, p.scales, prow, (int)p.I, kv_atoms, silu_tab,
                                     lane);
        else
            swiglu_mx_row<OUT, false>(src, out_row, p.scales, prow, (int)p.I, kv_atoms,
                                      silu_tab, lane);
    }
}

// ------------------------------------------------------ padded offsets

__global__ void padded_offsets_kernel(const uint32_t *ro, uint32_t *so, int G) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x;
    uint32_t carry = 0;
    if (lane == 0) so[0] = 0;
    for (int base = 0; base < G; base += 32) {
        int g = base + lane;
        uint32_t v = 0;
        if (g < G) {
            uint32_t a = ro[g], b = ro[g + 1];
            v = b > a ? ((b - a + 127u) & ~127u) : 0u;
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
            if (lane >= o) v += t;
        }
        if (g < G) so[g + 1] = carry + v;
        carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
}

}  // namespace

// ----------------------------------------------------------------- host

cudaError_t launch_amax_scale(const void *in, int64_t stride, int64_t K, const GroupArgs &g,
                              const Gather &gt, float *tensor_scale_out, uint32_t *err,
                              cudaStream_t s) {
    uint32_t *bits = reinterpret_cast<uint32_t *>(tensor_scale_out);
    const unsigned eblocks = (unsigned)((g.num_experts + 255) / 256);
    cudaError_t e = launch_pdl(zero_words_kernel, eblocks, 256, 0, s, bits, (int)g.num_experts);
    if (e != cudaSuccess) return e;
    if (g.total_rows > 0) {
        // one row per warp in small CTAs on small inputs (more, shorter CTAs
        // to fill the GPU), MOEQ_A_RPW rows per warp on large ones
        const bool large = g.total_rows >= 65536;
        const int rows_per_warp = large ? MOEQ_A_RPW : 1;
        const int cta_warps = large ? MOEQ_A_WARPS : MOEQ_A_WARPS_SMALL;
        int64_t warps = (g.total_rows + rows_per_warp - 1) / rows_per_warp;
        int64_t blocks = (warps + cta_warps - 1) / cta_warps;
        auto kern = large ? amax_kernel<MOEQ_A_WARPS, MOEQ_A_MINB>
                          : amax_kernel<MOEQ_A_WARPS_SMALL, MOEQ_A_MINB>;
        e = launch_pdl(kern, (unsigned)blocks, cta_warps * 32, 0, s,
                       reinterpret_cast<const uint16_t *>(in), stride, K, g, gt, bits, err,
                       rows_per_warp);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(amax_finalize_kernel, eblocks, 256, 0, s, bits, (int)g.num_experts);
}

cudaError_t launch_amax_scale_topk(const void *in, int64_t stride, int64_t K, int64_t num_tokens,
                                   const int32_t *topk_ids, int top_k, int num_experts,
                                   float *tensor_scale_out, uint32_t *err, cudaStream_t s) {
    uint32_t *bits = reinterpret_cast<uint32_t *>(tensor_scale_out);
    const unsigned eblocks = (unsigned)((num_experts + 255) / 256);
    cudaError_t e = launch_pdl(zero_words_kernel, eblocks, 256, 0, s, bits, num_experts);
    if (e != cudaSuccess) return e;
    if (num_tokens > 0) {
        const int rows_per_warp = num_tokens >= 65536 ? MOEQ_A_RPW : 1;
        const int64_t warps = (num_tokens + rows_per_warp - 1) / rows_per_warp;
        const int64_t blocks = (warps + MOEQ_A_WARPS - 1) / MOEQ_A_WARPS;
        e = launch_pdl(amax_topk_kernel, (unsigned)blocks, MOEQ_A_WARPS * 32, 0, s,
                       reinterpret_cast<const uint16_t *>(in), stride, K, num_tokens, topk_ids,
                       top_k, num_experts, bits, err, rows_per_warp);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(amax_finalize_kernel, eblocks, 256, 0, s, bits, num_experts);
}

cudaError_t launch_quantize(int fmt, const void *in, int64_t stride, int64_t K, uint8_t *out,
                            uint8_t *scales, const float *tensor_scale, const GroupArgs &g,
                            const Gather &gt, uint32_t *err, cudaStream_t s) {
    QuantParams p{reinterpret_cast<const uint16_t *>(in), stride, K, out, scales, tensor_scale,
                  g, gt, err};
    int64_t blocks = (g.scale_rows_total + kQWarps - 1) / kQWarps;
    if (blocks == 0) return cudaSuccess;
    // 256-bit loads need every row start 32-byte aligned
    const bool a32 = (reinterpret_cast<uintptr_t>(in) % 32 == 0) && (stride % 16 == 0);
    void (*kern)(QuantParams) =
        fmt == 0 ? (a32 ? quantize_kernel<0, true> : quantize_kernel<0, false>)
        : fmt == 1 ? (a32 ? quantize_kernel<1, true> : quantize_kernel<1, false>)
                   : (a32 ? quantize_kernel<2, true> : quantize_kernel<2, false>);
    return launch_pdl(kern, (unsigned)blocks, kQWarps * 32, 0, s, p);
}

cudaError_t launch_quantize_topk(int fmt, const void *in, int64_t stride, int64_t K,
                                 int64_t num_tokens, const int32_t *topk_ids, int top_k,
                                 const int32_t *dst_info, const uint32_t *row_offsets,
                                 const uint32_t *scales_offsets, const float *tensor_scale,
                                 int num_experts, int64_t total_rows, int64_t scale_rows_total,
                                 uint8_t *out, uint8_t *scales, uint32_t *err, cudaStream_t s) {
    const int64_t kv_atoms = K / (fmt == 0 ? 16 : 32) / 4;
    cudaError_t e = launch_pdl(zero_padding_scale_rows_kernel, (unsigned)num_experts, 256, 0, s,
                               row_offsets, scales_offsets, num_experts, total_rows,
                               scale_rows_total, kv_atoms, scales, err);
    if (e != cudaSuccess || num_tokens == 0) return e;
    TopkQuantParams p{reinterpret_cast<const uint16_t *>(in), stride, K, num_tokens, topk_ids,
                      dst_info, top_k, num_experts, row_offsets, scales_offsets, tensor_scale,
                      total_rows, scale_rows_total, out, scales, err};
    const int64_t blocks = (num_tokens + kQWarps - 1) / kQWarps;
    const bool a32 = (reinterpret_cast<uintptr_t>(in) % 32 == 0) && (stride % 16 == 0);
    void (*kern)(TopkQuantParams) =
        fmt == 0 ? (a32 ? quantize_topk_kernel<0, true> : quantize_topk_kernel<0, false>)
        : fmt == 1 ? (a32 ? quantize_topk_kernel<1, true> : quantize_topk_kernel<1, false>)
                   : (a32 ? quantize_topk_kernel<2, true> : quantize_topk_kernel<2, false>);
    return launch_pdl(kern, (unsigned)blocks, kQWarps * 32, 0, s, p);
}

cudaError_t launch_padded_offsets(const uint32_t *row_offsets, uint32_t *scales_offsets,
                                  int32_t num_groups, cudaStream_t s) {
    return launch_pdl(padded_offsets_kernel, 1, 32, 0, s, row_offsets, scales_offsets,
                      (int)num_groups);
}

cudaError_t launch_swiglu_quantize(int out_fmt, uint8_t *c_q, uint8_t *c_sf, const void *y,
                                   int64_t I, const float *out_tensor_scale, const GroupArgs &g,
                                   uint32_t *err, cudaStream_t s) {
    SwigluParams p{reinterpret_cast<const uint16_t *>(y), I, c_q, c_sf, out_tensor_scale, g, err};
    if (g.scale_rows_total == 0) return cudaSuccess;
    void (*kern)(SwigluParams) = out_fmt == 0   ? swiglu_nvfp4_kernel
                                 : out_fmt == 1 ? swiglu_mx_kernel<1>
                                                : swiglu_mx_kernel<2>;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    // per device: the SM count, and the opt-in for the table's dynamic shared
    // memory (static + dynamic exceed the default 48 KB), set once per kernel
    static std::atomic<int> sm_cache[kMaxDevices];
    static std::atomic<int> attr_cache[3][kMaxDevices];
    const int sms = cached_per_device(sm_cache, dev, [dev]() {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    });
    const int ok = cached_per_device(attr_cache[out_fmt], dev, [kern]() {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSiluTableBytes) == cudaSuccess ? 1 : 0;
    });
    if (!ok) return cudaErrorInvalidValue;
    const int64_t per_cta = (int64_t)kSWarps * MOEQ_SN_RPW;
    const int64_t blocks = std::min<int64_t>((g.scale_rows_total + per_cta - 1) / per_cta,
                                             (int64_t)sms * MOEQ_SN_MINB);
    return launch_pdl(kern, (unsigned)blocks, kSWarps * 32, kSiluTableBytes, s, p);
}

}  // namespace moeq
