// Internal launch interface between the C ABI (api.cu) and the kernel
// translation units.  Host-only declarations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace moeq {

// Per-device launch set-up (SM counts, kernel attributes already applied,
// occupancy answers) is computed once per device and cached.  The library
// may be called from several host threads at once, so every cache entry is
// an atomic, read without a lock and filled under launch_setup_mutex().
constexpr int kMaxDevices = 64;
std::mutex &launch_setup_mutex();

// cache[dev], filled once by fill() (a non-zero value; 0 means the set-up
// failed and leaves the entry empty, so a later call retries).
template <class T, class F>
T cached_per_device(std::atomic<T> (&cache)[kMaxDevices], int dev, F fill) {
    T v = cache[dev].load(std::memory_order_acquire);
    if (v) return v;
    std::lock_guard<std::mutex> lock(launch_setup_mutex());
    v = cache[dev].load(std::memory_order_relaxed);
    if (!v) {
        v = fill();
        if (v) cache[dev].store(v, std::memory_order_release);
    }
    return v;
}

struct GroupArgs {
    const uint32_t *row_offsets;     // [G+1]
    const uint32_t *scales_offsets;  // [G+1] or null
    const int32_t *expert_ids;       // [G]
    int32_t num_groups;
    int32_t num_experts;
    int64_t total_rows;
    int64_t scale_rows_total;
};

// Optional row gather of the streaming kernels: quantized row t reads input
// row indices[t] / divisor (in_rows input rows); indices == null: row t.
struct Gather {
    const int32_t *indices;
    int32_t divisor;
    int64_t in_rows;
};

cudaError_t launch_amax_scale(const void *in, int64_t stride, int64_t K, const GroupArgs &g,
                              const Gather &gt, float *tensor_scale_out, uint32_t *err,
                              cudaStream_t s);

// Per-expert tensor scales from tokens and their top-k ids (each token read once).
cudaError_t launch_amax_scale_topk(const void *in, int64_t stride, int64_t K, int64_t num_tokens,
                                   const int32_t *topk_ids, int top_k, int num_experts,
                                   float *tensor_scale_out, uint32_t *err, cudaStream_t s);

cudaError_t launch_quantize(int fmt, const void *in, int64_t stride, int64_t K, uint8_t *out,
                            uint8_t *scales, const float *tensor_scale, const GroupArgs &g,
                            const Gather &gt, uint32_t *err, cudaStream_t s);

// Token-major quantization of routed tokens (each token read once, written
// to every routed row dst_info[t * top_k + j]); top_k <= kTopkQuantMax.
constexpr int kTopkQuantMax = 8;
cudaError_t launch_quantize_topk(int fmt, const void *in, int64_t stride, int64_t K,
                                 int64_t num_tokens, const int32_t *topk_ids, int top_k,
                                 const int32_t *dst_info, const uint32_t *row_offsets,
                                 const uint32_t *scales_offsets, const float *tensor_scale,
                                 int num_experts, int64_t total_rows, int64_t scale_rows_total,
                                 uint8_t *out, uint8_t *scales, uint32_t *err, cudaStream_t s);

cudaError_t launch_padded_offsets(const uint32_t *row_offsets, uint32_t *scales_offsets,
                                  int32_t num_groups, cudaStream_t s);

// out_fmt: 0 NVFP4 (out_tensor_scale required), 1 MXFP4, 2 MXFP8.
cudaError_t launch_swiglu_quantize(int out_fmt, uint8_t *c_q, uint8_t *c_sf, const void *y,
                                   int64_t I, const float *out_tensor_scale, const GroupArgs &g,
                                   uint32_t *err, cudaStream_t s);

// Weight-preparation layout kernels (layout.cu).
cudaError_t launch_sf_swizzle(uint8_t *tiled, const uint8_t *logical, int64_t batch, int64_t rows,
                              int64_t kv, cudaStream_t s);
cudaError_t launch_sf_unswizzle(uint8_t *logical, const uint8_t *tiled, int64_t batch,
                                int64_t rows, int64_t kv, cudaStream_t s);
cudaError_t launch_interleave_rows(uint8_t *out, const uint8_t *gate, const uint8_t *up,
                                   int64_t batch, int64_t rows, int64_t row_bytes,
                                   cudaStream_t s);

// Routing of top-k choices to expert groups (route.cu); at most
// kRouteMaxExperts experts.  slot_rows > 0: scales_offsets[e] = e * slot_rows,
// else the padded prefix; scales_offsets may be null.
constexpr int kRouteMaxExperts = 1024;
cudaError_t launch_route_topk(const int32_t *topk_ids, int64_t num_choices, int num_experts,
                              uint32_t *row_offsets, int32_t *expert_ids, int32_t *src_info,
                              int32_t *dst_info, uint32_t *scales_offsets, int slot_rows,
                              uint32_t *err, cudaStream_t s);

// Grouped GEMMs.  kind: 0 = FP8 rowwise, 1 = NVFP4 block-scaled,
// 2 = MXFP8 block-scaled, 3 = MXFP4 block-scaled.  epi: 0 = bf16 out,
// 1 = fused SwiGLU + NVFP4, 2 = fused SwiGLU + MX in the mainloop's format.
struct GemmArgs {
    int kind;
    int epi;
    GroupArgs groups;
    int64_t N, K;
    const uint8_t *a, *b;
    const float *a_scales, *b_scales;      // FP8 rowwise
    const uint8_t *a_sf, *b_sf;            // block-scaled
    const float *expert_scales;            // block-scaled (null = 1)
    const float *out_tensor_scale;         // fused SwiGLU + NVFP4
    const uint16_t *row_scales;            // fused SwiGLU + NVFP4: bf16 per row, or null
    void *c;                               // bf16 out
    uint8_t *c_packed, *c_sf;              // fused SwiGLU out
    int32_t max_tokens_per_expert;
    uint32_t *err;
};

// Returns cudaErrorNotSupported for shapes without a built kernel.
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s);

// Maximum number of groups the GEMM scheduler accepts.
constexpr int kMaxGroups = 1024;

}  // namespace moeq
