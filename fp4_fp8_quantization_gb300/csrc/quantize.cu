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
// (grouped_quantize with padded scale alignment; fused_silu_quantize).
#include "common.cuh"
#include "launch.h"

namespace moeq {

namespace {

constexpr int kWarpsPerCta = 8;

// Checks one group's offsets / expert id; returns true if it can be used.
__device__ __forceinline__ bool group_ok(const GroupArgs &g, int gi, uint32_t *err,
                                         bool need_scales) {
    uint32_t r0 = __ldg(g.row_offsets + gi), r1 = __ldg(g.row_offsets + gi + 1);
    int e = __ldg(g.expert_ids + gi);
    if (r1 < r0 || (int64_t)r1 > g.total_rows) {
        set_error(err, MOEQ_DEVERR_BAD_OFFSETS);
        return false;
    }
    if (e < 0 || e >= g.num_experts) {
        set_error(err, MOEQ_DEVERR_BAD_EXPERT);
        return false;
    }
    if (need_scales) {
        uint32_t s0 = __ldg(g.scales_offsets + gi), s1 = __ldg(g.scales_offsets + gi + 1);
        uint32_t need = (r1 - r0 + 127u) & ~127u;
        if ((s0 & 127u) || s1 < s0 || s1 - s0 < need || (int64_t)s1 > g.scale_rows_total) {
            set_error(err, MOEQ_DEVERR_SCALE_ROWS);
            return false;
        }
    }
    return true;
}

// Maps logical scale row p to its group: returns g, or -1 when p lies in no
// group's scale range (or the group is invalid).
__device__ __forceinline__ int scale_row_group(const GroupArgs &g, uint32_t p, uint32_t *err) {
    int G = g.num_groups;
    uint32_t first = __ldg(g.scales_offsets), last = __ldg(g.scales_offsets + G);
    if (p < first || p >= last) return -1;
    int gi = upper_bound_minus1(g.scales_offsets, G, p);
    if (p >= __ldg(g.scales_offsets + gi + 1)) return -1;
    return group_ok(g, gi, err, true) ? gi : -1;
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

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&x)[8]) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
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

__global__ void __launch_bounds__(256) amax_kernel(const uint16_t *__restrict__ in,
                                                   int64_t stride, int64_t K, GroupArgs g,
                                                   uint32_t *__restrict__ amax_bits,
                                                   uint32_t *err, int rows_per_warp) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t row_begin = warp_id * rows_per_warp;
    const int G = g.num_groups;
    const uint32_t first = __ldg(g.row_offsets), last = __ldg(g.row_offsets + G);
    int cur_e = -1;
    uint32_t cur_m = 0;
    for (int64_t i = 0; i < rows_per_warp; ++i) {
        int64_t row = row_begin + i;
        if (row >= g.total_rows) break;
        if (row < first || row >= last) continue;
        int gi = upper_bound_minus1(g.row_offsets, G, (uint32_t)row);
        if (row >= __ldg(g.row_offsets + gi + 1) || !group_ok(g, gi, err, false)) continue;
        int e = __ldg(g.expert_ids + gi);
        const uint4 *src = reinterpret_cast<const uint4 *>(in + row * stride);
        uint32_t m = 0;
        const int64_t n16 = K / 8;
        int64_t c = lane;
        for (; c + 7 * 32 < n16; c += 8 * 32) {  // 8 independent loads in flight
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = ld_stream(src + c + u * 32);
#pragma unroll
            for (int u = 0; u < 8; ++u) m = max(m, bf16_abs_max8(v[u]));
        }
        for (; c < n16; c += 32) m = max(m, bf16_abs_max8(ld_stream(src + c)));
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (e != cur_e) {
            if (cur_e >= 0 && lane == 0 && cur_m) atomicMax(amax_bits + cur_e, cur_m << 16);
            cur_e = e;
            cur_m = 0;
        }
        cur_m = max(cur_m, m);
    }
    if (cur_e >= 0 && lane == 0 && cur_m) atomicMax(amax_bits + cur_e, cur_m << 16);
}

// amax (fp32 bits of a bf16 value) -> s = amax / 2688, or 1 for amax == 0.
__global__ void amax_finalize_kernel(uint32_t *buf, int E) {
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
    uint32_t *err;
};

// fmt: 0 NVFP4, 1 MXFP4, 2 MXFP8.  One warp per logical scale row.
template <int FMT>
__global__ void __launch_bounds__(256) quantize_kernel(QuantParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t prow = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (prow >= p.g.scale_rows_total) return;
    const int gi = scale_row_group(p.g, (uint32_t)prow, p.err);
    if (gi < 0) return;
    constexpr int V = FMT == 0 ? 16 : 32;
    const int64_t kv_atoms = p.K / V / 4;
    const uint32_t r0 = __ldg(p.g.row_offsets + gi);
    const uint32_t rg = __ldg(p.g.row_offsets + gi + 1) - r0;
    const uint32_t local = (uint32_t)prow - __ldg(p.g.scales_offsets + gi);
    if (local >= rg) {  // padding row of this group (up to the next multiple of 128)
        if (local < ((rg + 127u) & ~127u)) zero_scale_row(p.scales, prow, kv_atoms, lane);
        return;
    }
    const int64_t row = (int64_t)r0 + local;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.in + row * p.stride);
    float inv = 0.0f;
    if (FMT == 0) inv = __fdiv_rn(1.0f, __ldg(p.tensor_scale + __ldg(p.g.expert_ids + gi)));
    // 256 elements per warp step; with K % 256 == 128 the last step has
    // only lanes 0..15 active (they still take part in the shuffles).
    const int nchunks = (int)((p.K + 255) / 256);
    const int lanes_last = (int)((p.K / 8) - (int64_t)(nchunks - 1) * 32);
    constexpr int U = 8;  // 8 x 16 bytes in flight per lane
    for (int c0 = 0; c0 < nchunks; c0 += U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (c0 + u < nchunks && (c0 + u < nchunks - 1 || lane < lanes_last))
                v[u] = ld_stream(src + (int64_t)(c0 + u) * 32 + lane);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u;
            if (c >= nchunks) break;
            const bool active = c < nchunks - 1 || lane < lanes_last;
            float x[8];
            bf16x8_to_f32(v[u], x);
            uint32_t mb = bf16_abs_max8(v[u]);
            if (FMT == 0) {
                // block = 16 elements = lanes (2i, 2i+1)
                mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
                Nvfp4Scale s = nvfp4_block_scale(bf16_bits_to_f32(mb), inv);
                uint32_t codes = nvfp4_codes8(x, s.r);
                uint32_t word = gather4(s.code, lane, 2);
                if (!active) continue;
                reinterpret_cast<uint32_t *>(p.out + row * (p.K / 2))[c * 32 + lane] = codes;
                if ((lane & 7) == 0)
                    *reinterpret_cast<uint32_t *>(
                        p.scales + sf_word_offset(prow, c * 4 + (lane >> 3), kv_atoms)) = word;
            } else {
                // block = 32 elements = lanes (4i .. 4i+3)
                mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
                mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
                constexpr int emax = FMT == 2 ? 8 : 2;
                uint32_t code = 0;
                float y[8];
                if (mb == 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = 0.0f;
                } else {
                    int cs = bf16_floor_log2(mb) - emax + 127;
                    cs = min(max(cs, 0), 254);
                    code = (uint32_t)cs;
                    float f = __uint_as_float((uint32_t)(254 - cs) << 23);  // 2^(127-c)
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(x[i], f);
                }
                uint32_t word = gather4(code, lane, 4);
                if (!active) continue;
                if (FMT == 2) {
                    uint32_t lo = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
                    uint32_t hi = e4m3x2(y[4], y[5]) | (e4m3x2(y[6], y[7]) << 16);
                    if (mb == 0) lo = hi = 0u;
                    reinterpret_cast<uint2 *>(p.out + row * p.K)[c * 32 + lane] = make_uint2(lo, hi);
                } else {
                    uint32_t codes = (mb == 0) ? 0u : e2m1x8(y);
                    reinterpret_cast<uint32_t *>(p.out + row * (p.K / 2))[c * 32 + lane] = codes;
                }
                if ((lane & 15) == 0)
                    *reinterpret_cast<uint32_t *>(
                        p.scales + sf_word_offset(prow, c * 2 + (lane >> 4), kv_atoms)) = word;
            }
        }
    }
}

// --------------------------------------------- chained SwiGLU + NVFP4

struct SwigluParams {
    const uint16_t *y;   // [T, 2I] bf16
    int64_t I;
    uint8_t *out;        // [T, I/2]
    uint8_t *scales;
    const float *out_tensor_scale;
    GroupArgs g;
    uint32_t *err;
};

// One warp per logical scale row; a lane takes 8 (gate, up) pairs = 8 h
// values per 256-h step, so a 16-h block is held by lanes (2i, 2i+1).
__global__ void __launch_bounds__(256) swiglu_quantize_kernel(SwigluParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t prow = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (prow >= p.g.scale_rows_total) return;
    const int gi = scale_row_group(p.g, (uint32_t)prow, p.err);
    if (gi < 0) return;
    const int64_t kv_atoms = p.I / 64;
    const uint32_t r0 = __ldg(p.g.row_offsets + gi);
    const uint32_t rg = __ldg(p.g.row_offsets + gi + 1) - r0;
    const uint32_t local = (uint32_t)prow - __ldg(p.g.scales_offsets + gi);
    if (local >= rg) {
        if (local < ((rg + 127u) & ~127u)) zero_scale_row(p.scales, prow, kv_atoms, lane);
        return;
    }
    const int64_t row = (int64_t)r0 + local;
    const float inv = __fdiv_rn(1.0f, __ldg(p.out_tensor_scale + __ldg(p.g.expert_ids + gi)));
    const uint4 *src = reinterpret_cast<const uint4 *>(p.y + row * 2 * p.I);
    const int64_t nh = p.I;
    constexpr int U = 3;  // 256-h steps whose loads are issued together
    for (int64_t hb = 0; hb < nh; hb += 256 * U) {
      uint4 v[U][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t hl = hb + u * 256 + lane * 8;
        v[u][0] = v[u][1] = make_uint4(0u, 0u, 0u, 0u);
        if (hl < nh) {
            v[u][0] = ld_stream(src + hl / 4);
            v[u][1] = ld_stream(src + hl / 4 + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t h0 = hb + u * 256;
        if (h0 >= nh) break;
        const int64_t hl = h0 + lane * 8;          // first h of this lane
        const bool active = hl < nh;
        float h[8];
        if (active) {
            const uint4 v0 = v[u][0], v1 = v[u][1];
            uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float gate = bf16_bits_to_f32(w[i] & 0xFFFFu);
                float up = bf16_bits_to_f32(w[i] >> 16);
                h[i] = __fmul_rn(silu_spec(gate), up);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = 0.0f;
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(h[i]));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        Nvfp4Scale s = nvfp4_block_scale(m, inv);
        uint32_t codes = nvfp4_codes8(h, s.r);
        uint32_t word = gather4(s.code, lane, 2);
        if (active) {
            reinterpret_cast<uint32_t *>(p.out + row * (p.I / 2))[hl / 8] = codes;
            if ((lane & 7) == 0)
                *reinterpret_cast<uint32_t *>(
                    p.scales + sf_word_offset(prow, hl / 64, kv_atoms)) = word;
        }
      }
    }
}

// ------------------------------------------------------ padded offsets

__global__ void padded_offsets_kernel(const uint32_t *ro, uint32_t *so, int G) {
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
                              float *tensor_scale_out, uint32_t *err, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(tensor_scale_out, 0, sizeof(float) * g.num_experts, s);
    if (e != cudaSuccess) return e;
    if (g.total_rows > 0) {
        const int rows_per_warp = 4;
        int64_t warps = (g.total_rows + rows_per_warp - 1) / rows_per_warp;
        int64_t blocks = (warps + 7) / 8;
        amax_kernel<<<(unsigned)blocks, 256, 0, s>>>(
            reinterpret_cast<const uint16_t *>(in), stride, K, g,
            reinterpret_cast<uint32_t *>(tensor_scale_out), err, rows_per_warp);
    }
    amax_finalize_kernel<<<(g.num_experts + 255) / 256, 256, 0, s>>>(
        reinterpret_cast<uint32_t *>(tensor_scale_out), g.num_experts);
    return cudaGetLastError();
}

cudaError_t launch_quantize(int fmt, const void *in, int64_t stride, int64_t K, uint8_t *out,
                            uint8_t *scales, const float *tensor_scale, const GroupArgs &g,
                            uint32_t *err, cudaStream_t s) {
    QuantParams p{reinterpret_cast<const uint16_t *>(in), stride, K, out, scales, tensor_scale,
                  g, err};
    int64_t blocks = (g.scale_rows_total + kWarpsPerCta - 1) / kWarpsPerCta;
    if (blocks == 0) return cudaSuccess;
    if (fmt == 0)
        quantize_kernel<0><<<(unsigned)blocks, 256, 0, s>>>(p);
    else if (fmt == 1)
        quantize_kernel<1><<<(unsigned)blocks, 256, 0, s>>>(p);
    else
        quantize_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_padded_offsets(const uint32_t *row_offsets, uint32_t *scales_offsets,
                                  int32_t num_groups, cudaStream_t s) {
    padded_offsets_kernel<<<1, 32, 0, s>>>(row_offsets, scales_offsets, num_groups);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_quantize(uint8_t *c_packed, uint8_t *c_sf, const void *y, int64_t I,
                                   const float *out_tensor_scale, const GroupArgs &g,
                                   uint32_t *err, cudaStream_t s) {
    SwigluParams p{reinterpret_cast<const uint16_t *>(y), I, c_packed, c_sf, out_tensor_scale,
                   g, err};
    int64_t blocks = (g.scale_rows_total + kWarpsPerCta - 1) / kWarpsPerCta;
    if (blocks == 0) return cudaSuccess;
    swiglu_quantize_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace moeq
