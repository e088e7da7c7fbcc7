// C ABI of the moeq library: host-side argument validation, the device
// error word, and dispatch to the kernel launchers.  Every compute entry
// point only enqueues work on the caller's stream.
#include <stdint.h>

#include "../../include/moeq.h"
#include "common.cuh"
#include "launch.h"

namespace {

__device__ uint32_t g_device_error;

thread_local int t_last_cuda_error = 0;

// Address of the device error word on the current device (looked up once
// per device).
uint32_t *device_error_ptr() {
    static std::atomic<uint32_t *> cache[moeq::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= moeq::kMaxDevices) return nullptr;
    return moeq::cached_per_device(cache, dev, []() -> uint32_t * {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        return static_cast<uint32_t *>(p);
    });
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moeq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOEQ_OK;
    if (e == cudaErrorNotSupported) return MOEQ_ERR_UNSUPPORTED;
    t_last_cuda_error = (int)e;
    return MOEQ_ERR_CUDA;
}

// Common checks of the ragged-group description.
bool groups_ok(const uint32_t *offs, const int32_t *ids, int32_t num_experts,
               int32_t num_active_experts) {
    if (num_active_experts < 0 || num_experts <= 0) return false;
    if (num_active_experts > 0 && (!offs || !ids)) return false;
    return true;
}

moeq::GroupArgs make_groups(const uint32_t *ro, const uint32_t *so, const int32_t *ids,
                            int32_t G, int32_t E, int64_t rows, int64_t scale_rows) {
    moeq::GroupArgs g;
    g.row_offsets = ro;
    g.scales_offsets = so;
    g.expert_ids = ids;
    g.num_groups = G;
    g.num_experts = E;
    g.total_rows = rows;
    g.scale_rows_total = scale_rows;
    return g;
}

}  // namespace

std::mutex &moeq::launch_setup_mutex() {
    static std::mutex m;
    return m;
}

extern "C" {

const char *moeq_status_string(moeq_status s) {
    switch (s) {
        case MOEQ_OK: return "MOEQ_OK";
        case MOEQ_ERR_INVALID_ARG: return "MOEQ_ERR_INVALID_ARG";
        case MOEQ_ERR_UNSUPPORTED: return "MOEQ_ERR_UNSUPPORTED";
        case MOEQ_ERR_CUDA: return "MOEQ_ERR_CUDA";
        case MOEQ_ERR_DEVICE: return "MOEQ_ERR_DEVICE";
    }
    return "MOEQ_UNKNOWN_STATUS";
}

int moeq_last_cuda_error(void) { return t_last_cuda_error; }

moeq_status moeq_get_device_error(moeq_stream_t stream, uint32_t *bits) {
    if (!bits) return MOEQ_ERR_INVALID_ARG;
    uint32_t *p = device_error_ptr();
    if (!p) return cuda_status(cudaErrorInvalidDevice);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_status(e);
    *bits = v;
    return v ? MOEQ_ERR_DEVICE : MOEQ_OK;
}

moeq_status moeq_clear_device_error(moeq_stream_t stream) {
    uint32_t *p = device_error_ptr();
    if (!p) return cuda_status(cudaErrorInvalidDevice);
    return cuda_status(cudaMemsetAsync(p, 0, sizeof(uint32_t), stream));
}

moeq_status moeq_padded_scale_offsets(const uint32_t *row_offsets, uint32_t *scales_offsets,
                                      int32_t num_active_experts, moeq_stream_t stream) {
    if (num_active_experts < 0 || !row_offsets || !scales_offsets) return MOEQ_ERR_INVALID_ARG;
    return cuda_status(
        moeq::launch_padded_offsets(row_offsets, scales_offsets, num_active_experts, stream));
}

// Sizes of the layout helpers: products stay far below 2^62.
static bool layout_sizes_ok(int64_t batch, int64_t rows, int64_t cols) {
    const int64_t lim = (int64_t)1 << 40;
    return batch >= 0 && rows >= 0 && cols >= 0 && batch < lim && rows < lim && cols < lim &&
           (batch == 0 || rows == 0 || cols == 0 ||
            (double)batch * (double)(rows + 128) * (double)(cols + 4) < 4e18);
}

moeq_status moeq_sf_swizzle(uint8_t *tiled, const uint8_t *logical, int64_t batch, int64_t rows,
                            int64_t kv, moeq_stream_t stream) {
    if (!layout_sizes_ok(batch, rows, kv)) return MOEQ_ERR_INVALID_ARG;
    if (batch == 0 || rows == 0 || kv == 0) return MOEQ_OK;
    if (!tiled || !logical) return MOEQ_ERR_INVALID_ARG;
    return cuda_status(moeq::launch_sf_swizzle(tiled, logical, batch, rows, kv, stream));
}

moeq_status moeq_sf_unswizzle(uint8_t *logical, const uint8_t *tiled, int64_t batch,
                              int64_t rows, int64_t kv, moeq_stream_t stream) {
    if (!layout_sizes_ok(batch, rows, kv)) return MOEQ_ERR_INVALID_ARG;
    if (batch == 0 || rows == 0 || kv == 0) return MOEQ_OK;
    if (!tiled || !logical) return MOEQ_ERR_INVALID_ARG;
    return cuda_status(moeq::launch_sf_unswizzle(logical, tiled, batch, rows, kv, stream));
}

moeq_status moeq_interleave_gate_up(uint8_t *out, const uint8_t *gate, const uint8_t *up,
                                    int64_t batch, int64_t rows, int64_t row_bytes,
                                    moeq_stream_t stream) {
    if (!layout_sizes_ok(batch, 2 * rows, row_bytes)) return MOEQ_ERR_INVALID_ARG;
    if (batch == 0 || rows == 0 || row_bytes == 0) return MOEQ_OK;
    if (!out || !gate || !up) return MOEQ_ERR_INVALID_ARG;
    return cuda_status(
        moeq::launch_interleave_rows(out, gate, up, batch, rows, row_bytes, stream));
}

static moeq_status amax_impl(const void *in, int64_t in_row_stride, int64_t total_rows,
                             int64_t K, const uint32_t *row_offsets, const int32_t *expert_ids,
                             float *tensor_scale_out, int32_t num_experts,
                             int32_t num_active_experts, const moeq::Gather &gt,
                             moeq_stream_t stream) {
    if (!groups_ok(row_offsets, expert_ids, num_experts, num_active_experts))
        return MOEQ_ERR_INVALID_ARG;
    if (!tensor_scale_out || total_rows < 0 || K <= 0 || K % 8 || in_row_stride < K ||
        in_row_stride % 8)
        return MOEQ_ERR_INVALID_ARG;
    if (total_rows > 0 && (!in || !aligned16(in))) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(tensor_scale_out)) return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    moeq::GroupArgs g = make_groups(row_offsets, nullptr, expert_ids, num_active_experts,
                                    num_experts, num_active_experts ? total_rows : 0, 0);
    return cuda_status(
        moeq::launch_amax_scale(in, in_row_stride, K, g, gt, tensor_scale_out, err, stream));
}

static moeq_status quantize_impl(moeq_format fmt, const void *in, int64_t in_row_stride,
                                 int64_t total_rows, int64_t K, uint8_t *out, uint8_t *scales,
                                 int64_t scale_rows_total, const uint32_t *row_offsets,
                                 const uint32_t *scales_offsets, const int32_t *expert_ids,
                                 const float *tensor_scale, int32_t num_experts,
                                 int32_t num_active_experts, const moeq::Gather &gt,
                                 moeq_stream_t stream) {
    if (fmt != MOEQ_NVFP4 && fmt != MOEQ_MXFP4 && fmt != MOEQ_MXFP8) return MOEQ_ERR_INVALID_ARG;
    if (!groups_ok(row_offsets, expert_ids, num_experts, num_active_experts))
        return MOEQ_ERR_INVALID_ARG;
    if (total_rows < 0 || K <= 0 || K % 128 || in_row_stride < K || in_row_stride % 8 ||
        scale_rows_total < 0 || scale_rows_total % 128)
        return MOEQ_ERR_INVALID_ARG;
    if (fmt == MOEQ_NVFP4 && !tensor_scale) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts == 0 || total_rows == 0 || scale_rows_total == 0) return MOEQ_OK;
    if (!scales_offsets || !in || !out || !scales || !aligned16(in) || !aligned16(out) ||
        !aligned16(scales))
        return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    moeq::GroupArgs g = make_groups(row_offsets, scales_offsets, expert_ids, num_active_experts,
                                    num_experts, total_rows, scale_rows_total);
    return cuda_status(moeq::launch_quantize((int)fmt, in, in_row_stride, K, out, scales,
                                             tensor_scale, g, gt, err, stream));
}

static bool gather_ok(const int32_t *indices, int32_t indices_divisor, int64_t in_rows,
                      int64_t total_rows) {
    return indices_divisor >= 1 && in_rows >= 0 && (total_rows == 0 || indices);
}

moeq_status moeq_grouped_amax_scale(const void *in, int64_t in_row_stride, int64_t total_rows,
                                    int64_t K, const uint32_t *row_offsets,
                                    const int32_t *expert_ids, float *tensor_scale_out,
                                    int32_t num_experts, int32_t num_active_experts,
                                    moeq_stream_t stream) {
    const moeq::Gather none{nullptr, 1, total_rows};
    return amax_impl(in, in_row_stride, total_rows, K, row_offsets, expert_ids, tensor_scale_out,
                     num_experts, num_active_experts, none, stream);
}

moeq_status moeq_grouped_amax_scale_gather(const void *in, int64_t in_row_stride,
                                           int64_t in_rows, int64_t K,
                                           const int32_t *indices, int32_t indices_divisor,
                                           int64_t total_rows, const uint32_t *row_offsets,
                                           const int32_t *expert_ids, float *tensor_scale_out,
                                           int32_t num_experts, int32_t num_active_experts,
                                           moeq_stream_t stream) {
    if (!gather_ok(indices, indices_divisor, in_rows, total_rows)) return MOEQ_ERR_INVALID_ARG;
    if (in_rows == 0 && total_rows > 0 && num_active_experts > 0) return MOEQ_ERR_INVALID_ARG;
    const moeq::Gather gt{indices, indices_divisor, in_rows};
    return amax_impl(in, in_row_stride, total_rows, K, row_offsets, expert_ids, tensor_scale_out,
                     num_experts, num_active_experts, gt, stream);
}

moeq_status moeq_grouped_quantize(moeq_format fmt, const void *in, int64_t in_row_stride,
                                  int64_t total_rows, int64_t K, uint8_t *out, uint8_t *scales,
                                  int64_t scale_rows_total, const uint32_t *row_offsets,
                                  const uint32_t *scales_offsets, const int32_t *expert_ids,
                                  const float *tensor_scale, int32_t num_experts,
                                  int32_t max_tokens_per_expert, int32_t num_active_experts,
                                  moeq_stream_t stream) {
    (void)max_tokens_per_expert;
    const moeq::Gather none{nullptr, 1, total_rows};
    return quantize_impl(fmt, in, in_row_stride, total_rows, K, out, scales, scale_rows_total,
                         row_offsets, scales_offsets, expert_ids, tensor_scale, num_experts,
                         num_active_experts, none, stream);
}

moeq_status moeq_grouped_quantize_gather(moeq_format fmt, const void *in, int64_t in_row_stride,
                                         int64_t in_rows, int64_t K, const int32_t *indices,
                                         int32_t indices_divisor, int64_t total_rows,
                                         uint8_t *out, uint8_t *scales, int64_t scale_rows_total,
                                         const uint32_t *row_offsets,
                                         const uint32_t *scales_offsets,
                                         const int32_t *expert_ids, const float *tensor_scale,
                                         int32_t num_experts, int32_t max_tokens_per_expert,
                                         int32_t num_active_experts, moeq_stream_t stream) {
    (void)max_tokens_per_expert;
    if (!gather_ok(indices, indices_divisor, in_rows, total_rows)) return MOEQ_ERR_INVALID_ARG;
    if (in_rows == 0 && total_rows > 0 && num_active_experts > 0) return MOEQ_ERR_INVALID_ARG;
    const moeq::Gather gt{indices, indices_divisor, in_rows};
    return quantize_impl(fmt, in, in_row_stride, total_rows, K, out, scales, scale_rows_total,
                         row_offsets, scales_offsets, expert_ids, tensor_scale, num_experts,
                         num_active_experts, gt, stream);
}

// ------------------------------------------------------------ dispatch

static moeq_status route_args_ok(const int32_t *topk_ids, int64_t num_tokens, int32_t top_k,
                                 int32_t num_experts, const uint32_t *row_offsets,
                                 const int32_t *expert_ids, const int32_t *src_info,
                                 const int32_t *dst_info, const uint32_t *scales_offsets,
                                 int32_t slot_rows) {
    if (num_tokens < 0 || top_k < 1 || num_experts < 1 || slot_rows < 0 || slot_rows % 128)
        return MOEQ_ERR_INVALID_ARG;
    if (num_experts > moeq::kRouteMaxExperts || num_tokens >= ((int64_t)1 << 31) / top_k)
        return MOEQ_ERR_UNSUPPORTED;
    if (!row_offsets || !expert_ids || !aligned16(row_offsets) || !aligned16(expert_ids))
        return MOEQ_ERR_INVALID_ARG;
    if (scales_offsets && !aligned16(scales_offsets)) return MOEQ_ERR_INVALID_ARG;
    if (dst_info && !aligned16(dst_info)) return MOEQ_ERR_INVALID_ARG;
    if (num_tokens > 0 &&
        (!topk_ids || !src_info || !aligned16(topk_ids) || !aligned16(src_info)))
        return MOEQ_ERR_INVALID_ARG;
    return MOEQ_OK;
}

moeq_status moeq_route_topk(const int32_t *topk_ids, int64_t num_tokens, int32_t top_k,
                            int32_t num_experts, uint32_t *row_offsets, int32_t *expert_ids,
                            int32_t *src_info, int32_t *dst_info, uint32_t *scales_offsets,
                            int32_t slot_rows, moeq_stream_t stream) {
    const moeq_status st = route_args_ok(topk_ids, num_tokens, top_k, num_experts, row_offsets,
                                         expert_ids, src_info, dst_info, scales_offsets,
                                         slot_rows);
    if (st != MOEQ_OK) return st;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    return cuda_status(moeq::launch_route_topk(topk_ids, num_tokens * top_k, num_experts,
                                               row_offsets, expert_ids, src_info, dst_info,
                                               scales_offsets, slot_rows, err, stream));
}

moeq_status moeq_grouped_amax_scale_topk(const void *tokens, int64_t token_stride,
                                         int64_t num_tokens, int64_t K, const int32_t *topk_ids,
                                         int32_t top_k, float *tensor_scale_out,
                                         int32_t num_experts, moeq_stream_t stream) {
    if (num_tokens < 0 || top_k < 1 || num_experts < 1 || K <= 0 || K % 8 ||
        token_stride < K || token_stride % 8 || !tensor_scale_out ||
        !aligned16(tensor_scale_out))
        return MOEQ_ERR_INVALID_ARG;
    if (num_tokens >= ((int64_t)1 << 31) / top_k) return MOEQ_ERR_UNSUPPORTED;
    if (num_tokens > 0 &&
        (!tokens || !topk_ids || !aligned16(tokens) || !aligned16(topk_ids)))
        return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    return cuda_status(moeq::launch_amax_scale_topk(tokens, token_stride, K, num_tokens, topk_ids,
                                                    top_k, num_experts, tensor_scale_out, err,
                                                    stream));
}

int64_t moeq_dispatch_scale_rows(int64_t num_tokens, int32_t top_k, int32_t num_experts,
                                 int32_t slot_rows) {
    if (num_tokens < 0 || top_k < 1 || num_experts < 1 || slot_rows < 0 ||
        num_tokens >= ((int64_t)1 << 31) / top_k)
        return -1;
    if (slot_rows > 0) return (int64_t)num_experts * slot_rows;
    // sum over experts of ceil(r_e / 128) * 128 <= sum (r_e + 127), a multiple of 128
    return (num_tokens * top_k + 127 * (int64_t)num_experts) / 128 * 128;
}

moeq_status moeq_quantize_topk(moeq_format fmt, const void *tokens, int64_t token_stride,
                               int64_t num_tokens, int64_t K, const int32_t *topk_ids,
                               int32_t top_k, const int32_t *dst_info,
                               const uint32_t *row_offsets, const uint32_t *scales_offsets,
                               const float *tensor_scale, int32_t num_experts, uint8_t *out,
                               uint8_t *scales, int64_t scale_rows_total, moeq_stream_t stream) {
    if (fmt != MOEQ_NVFP4 && fmt != MOEQ_MXFP4 && fmt != MOEQ_MXFP8) return MOEQ_ERR_INVALID_ARG;
    if (num_tokens < 0 || top_k < 1 || num_experts < 1 || K <= 0 || K % 128 ||
        token_stride < K || token_stride % 8 || scale_rows_total < 0 || scale_rows_total % 128)
        return MOEQ_ERR_INVALID_ARG;
    if (top_k > moeq::kTopkQuantMax || num_experts > moeq::kRouteMaxExperts ||
        num_tokens >= ((int64_t)1 << 31) / top_k)
        return MOEQ_ERR_UNSUPPORTED;
    if (fmt == MOEQ_NVFP4 && !tensor_scale) return MOEQ_ERR_INVALID_ARG;
    if (!row_offsets || !scales_offsets || !scales || !aligned16(scales)) return MOEQ_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!tokens || !topk_ids || !dst_info || !out || !aligned16(tokens) ||
                           !aligned16(topk_ids) || !aligned16(dst_info) || !aligned16(out)))
        return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    return cuda_status(moeq::launch_quantize_topk(
        (int)fmt, tokens, token_stride, K, num_tokens, topk_ids, top_k, dst_info, row_offsets,
        scales_offsets, tensor_scale, num_experts, num_tokens * top_k, scale_rows_total, out,
        scales, err, stream));
}

moeq_status moeq_dispatch_mxfp4(const void *tokens, int64_t token_stride, int64_t num_tokens,
                                int64_t hidden, const int32_t *topk_ids, int32_t top_k,
                                int32_t num_experts, uint8_t *out, uint8_t *scales,
                                int64_t scale_rows_total, uint32_t *row_offsets,
                                int32_t *expert_ids, int32_t *src_info, int32_t *dst_info,
                                uint32_t *scales_offsets, int32_t slot_rows,
                                moeq_stream_t stream) {
    moeq_status st = route_args_ok(topk_ids, num_tokens, top_k, num_experts, row_offsets,
                                   expert_ids, src_info, dst_info, scales_offsets, slot_rows);
    if (st != MOEQ_OK) return st;
    // every check of the quantization step before anything is launched
    if (!scales_offsets || hidden <= 0 || hidden % 128 || token_stride < hidden ||
        token_stride % 8 || scale_rows_total % 128 || !scales || !aligned16(scales) ||
        scale_rows_total < moeq_dispatch_scale_rows(num_tokens, top_k, num_experts, slot_rows))
        return MOEQ_ERR_INVALID_ARG;
    if (top_k > moeq::kTopkQuantMax) return MOEQ_ERR_UNSUPPORTED;
    if (num_tokens > 0 && (!tokens || !out || !dst_info || !aligned16(tokens) || !aligned16(out)))
        return MOEQ_ERR_INVALID_ARG;
    st = moeq_route_topk(topk_ids, num_tokens, top_k, num_experts, row_offsets, expert_ids,
                         src_info, dst_info, scales_offsets, slot_rows, stream);
    if (st != MOEQ_OK) return st;
    // token-major: each token read and quantized once, stored to its routed rows
    return moeq_quantize_topk(MOEQ_MXFP4, tokens, token_stride, num_tokens, hidden, topk_ids,
                              top_k, dst_info, row_offsets, scales_offsets, nullptr, num_experts,
                              out, scales, scale_rows_total, stream);
}

moeq_status moeq_grouped_matmul_rowwise_fp8(void *c, const uint8_t *a, const uint8_t *b,
                                            const float *a_scales, const float *b_scales,
                                            const uint32_t *a_offsets,
                                            const int32_t *expert_ids, int64_t total_tokens,
                                            int64_t N, int64_t K, int32_t num_experts,
                                            int32_t max_tokens_per_expert,
                                            int32_t num_active_experts, moeq_stream_t stream) {
    if (!groups_ok(a_offsets, expert_ids, num_experts, num_active_experts))
        return MOEQ_ERR_INVALID_ARG;
    if (total_tokens < 0 || N <= 0 || K <= 0 || K % 128 || N % 16) return MOEQ_ERR_INVALID_ARG;
    if (total_tokens >= (int64_t)1 << 31 || N >= (int64_t)1 << 31 || K >= (int64_t)1 << 31)
        return MOEQ_ERR_UNSUPPORTED;
    if (num_active_experts > moeq::kMaxGroups) return MOEQ_ERR_UNSUPPORTED;
    if (!b || !b_scales || !aligned16(b) || !aligned16(b_scales)) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts == 0 || total_tokens == 0) return MOEQ_OK;
    if (!c || !a || !a_scales || !aligned16(c) || !aligned16(a) || !aligned16(a_scales))
        return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    moeq::GemmArgs ga = {};
    ga.kind = 0;
    ga.epi = 0;
    ga.groups = make_groups(a_offsets, nullptr, expert_ids, num_active_experts, num_experts,
                            total_tokens, 0);
    ga.N = N;
    ga.K = K;
    ga.a = a;
    ga.b = b;
    ga.a_scales = a_scales;
    ga.b_scales = b_scales;
    ga.c = c;
    ga.max_tokens_per_expert = max_tokens_per_expert;
    ga.err = err;
    return cuda_status(moeq::launch_gemm(ga, stream));
}

static moeq_status blockscaled_common(moeq_format fmt, int epi, const uint8_t *a,
                                      const uint8_t *a_sf, const uint8_t *b, const uint8_t *b_sf,
                                      const uint32_t *a_offsets,
                                      const uint32_t *a_scales_offsets,
                                      const int32_t *expert_ids, int64_t total_tokens,
                                      int64_t scale_rows_total, int64_t N, int64_t K,
                                      int32_t num_experts, int32_t num_active_experts,
                                      moeq::GemmArgs *ga) {
    if (!groups_ok(a_offsets, expert_ids, num_experts, num_active_experts))
        return MOEQ_ERR_INVALID_ARG;
    if (fmt != MOEQ_NVFP4 && fmt != MOEQ_MXFP4 && fmt != MOEQ_MXFP8) return MOEQ_ERR_INVALID_ARG;
    if (total_tokens < 0 || N <= 0 || K <= 0 || N % 128 || scale_rows_total < 0 ||
        scale_rows_total % 128)
        return MOEQ_ERR_INVALID_ARG;
    if (fmt == MOEQ_MXFP8 ? (K % 128) : (K % 256)) return MOEQ_ERR_INVALID_ARG;
    if (total_tokens >= (int64_t)1 << 31 || N >= (int64_t)1 << 31 || K >= (int64_t)1 << 31)
        return MOEQ_ERR_UNSUPPORTED;
    if (num_active_experts > moeq::kMaxGroups) return MOEQ_ERR_UNSUPPORTED;
    if (!b || !b_sf || !aligned16(b) || !aligned16(b_sf)) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts > 0 && !a_scales_offsets) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts > 0 && total_tokens > 0 &&
        (!a || !a_sf || !aligned16(a) || !aligned16(a_sf)))
        return MOEQ_ERR_INVALID_ARG;
    *ga = moeq::GemmArgs{};
    ga->kind = fmt == MOEQ_NVFP4 ? 1 : (fmt == MOEQ_MXFP8 ? 2 : 3);
    ga->epi = epi;
    ga->groups = make_groups(a_offsets, a_scales_offsets, expert_ids, num_active_experts,
                             num_experts, total_tokens, scale_rows_total);
    ga->N = N;
    ga->K = K;
    ga->a = a;
    ga->b = b;
    ga->a_sf = a_sf;
    ga->b_sf = b_sf;
    return MOEQ_OK;
}

moeq_status moeq_grouped_matmul_blockscaled(
    moeq_format fmt, void *c, const uint8_t *a, const uint8_t *a_sf, const uint8_t *b,
    const uint8_t *b_sf, const float *expert_scales, const uint32_t *a_offsets,
    const uint32_t *a_scales_offsets, const int32_t *expert_ids, int64_t total_tokens,
    int64_t scale_rows_total, int64_t N, int64_t K, int32_t num_experts,
    int32_t max_tokens_per_expert, int32_t num_active_experts, moeq_stream_t stream) {
    moeq::GemmArgs ga;
    moeq_status st =
        blockscaled_common(fmt, 0, a, a_sf, b, b_sf, a_offsets, a_scales_offsets, expert_ids,
                           total_tokens, scale_rows_total, N, K, num_experts,
                           num_active_experts, &ga);
    if (st != MOEQ_OK) return st;
    if (fmt == MOEQ_NVFP4 && !expert_scales) return MOEQ_ERR_INVALID_ARG;
    if (expert_scales && !aligned16(expert_scales)) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts == 0 || total_tokens == 0) return MOEQ_OK;
    if (!c || !aligned16(c)) return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    ga.expert_scales = expert_scales;
    ga.c = c;
    ga.max_tokens_per_expert = max_tokens_per_expert;
    ga.err = err;
    return cuda_status(moeq::launch_gemm(ga, stream));
}

static moeq_status swiglu_quantize_impl(int out_fmt, uint8_t *c_q, uint8_t *c_sf, const void *y,
                                        const float *out_tensor_scale, const uint32_t *a_offsets,
                                        const uint32_t *a_scales_offsets,
                                        const int32_t *expert_ids, int64_t total_tokens,
                                        int64_t scale_rows_total, int64_t I, int32_t num_experts,
                                        int32_t num_active_experts, moeq_stream_t stream) {
    if (!groups_ok(a_offsets, expert_ids, num_experts, num_active_experts))
        return MOEQ_ERR_INVALID_ARG;
    if (total_tokens < 0 || I <= 0 || I % (out_fmt == 0 ? 64 : 128) || scale_rows_total < 0 ||
        scale_rows_total % 128)
        return MOEQ_ERR_INVALID_ARG;
    if (out_fmt == 0 && !out_tensor_scale) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts == 0 || total_tokens == 0 || scale_rows_total == 0) return MOEQ_OK;
    if (!a_scales_offsets || !y || !c_q || !c_sf || !aligned16(y) || !aligned16(c_q) ||
        !aligned16(c_sf))
        return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    moeq::GroupArgs g = make_groups(a_offsets, a_scales_offsets, expert_ids, num_active_experts,
                                    num_experts, total_tokens, scale_rows_total);
    return cuda_status(moeq::launch_swiglu_quantize(out_fmt, c_q, c_sf, y, I, out_tensor_scale, g,
                                                    err, stream));
}

moeq_status moeq_swiglu_quantize(uint8_t *c_packed, uint8_t *c_sf, const void *y,
                                 const float *out_tensor_scale, const uint32_t *a_offsets,
                                 const uint32_t *a_scales_offsets, const int32_t *expert_ids,
                                 int64_t total_tokens, int64_t scale_rows_total, int64_t I,
                                 int32_t num_experts, int32_t max_tokens_per_expert,
                                 int32_t num_active_experts, moeq_stream_t stream) {
    (void)max_tokens_per_expert;
    return swiglu_quantize_impl(0, c_packed, c_sf, y, out_tensor_scale, a_offsets,
                                a_scales_offsets, expert_ids, total_tokens, scale_rows_total, I,
                                num_experts, num_active_experts, stream);
}

moeq_status moeq_swiglu_quantize_mx(moeq_format fmt, uint8_t *c_q, uint8_t *c_sf, const void *y,
                                    const uint32_t *a_offsets, const uint32_t *a_scales_offsets,
                                    const int32_t *expert_ids, int64_t total_tokens,
                                    int64_t scale_rows_total, int64_t I, int32_t num_experts,
                                    int32_t max_tokens_per_expert, int32_t num_active_experts,
                                    moeq_stream_t stream) {
    (void)max_tokens_per_expert;
    if (fmt != MOEQ_MXFP4 && fmt != MOEQ_MXFP8) return MOEQ_ERR_INVALID_ARG;
    return swiglu_quantize_impl((int)fmt, c_q, c_sf, y, nullptr, a_offsets, a_scales_offsets,
                                expert_ids, total_tokens, scale_rows_total, I, num_experts,
                                num_active_experts, stream);
}

moeq_status moeq_grouped_matmul_swiglu(
    uint8_t *c_packed, uint8_t *c_sf, const uint8_t *a, const uint8_t *a_sf, const uint8_t *b,
    const uint8_t *b_sf, const float *expert_scales, const float *out_tensor_scale,
    const void *a_row_scales, const uint32_t *a_offsets, const uint32_t *a_scales_offsets,
    const int32_t *expert_ids, int64_t total_tokens, int64_t scale_rows_total, int64_t I,
    int64_t K, int32_t num_experts, int32_t max_tokens_per_expert, int32_t num_active_experts,
    moeq_stream_t stream) {
    if (I <= 0 || I % 64) return MOEQ_ERR_INVALID_ARG;
    moeq::GemmArgs ga;
    moeq_status st = blockscaled_common(MOEQ_NVFP4, 1, a, a_sf, b, b_sf, a_offsets,
                                        a_scales_offsets, expert_ids, total_tokens,
                                        scale_rows_total, 2 * I, K, num_experts,
                                        num_active_experts, &ga);
    if (st != MOEQ_OK) return st;
    if (!expert_scales || !out_tensor_scale) return MOEQ_ERR_INVALID_ARG;
    if (a_row_scales && !aligned16(a_row_scales)) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts == 0 || total_tokens == 0) return MOEQ_OK;
    if (!c_packed || !c_sf || !aligned16(c_packed) || !aligned16(c_sf))
        return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    ga.expert_scales = expert_scales;
    ga.out_tensor_scale = out_tensor_scale;
    ga.row_scales = static_cast<const uint16_t *>(a_row_scales);
    ga.c_packed = c_packed;
    ga.c_sf = c_sf;
    ga.max_tokens_per_expert = max_tokens_per_expert;
    ga.err = err;
    return cuda_status(moeq::launch_gemm(ga, stream));
}

moeq_status moeq_grouped_matmul_swiglu_mx(
    moeq_format fmt, uint8_t *c_q, uint8_t *c_sf, const uint8_t *a, const uint8_t *a_sf,
    const uint8_t *b, const uint8_t *b_sf, const float *expert_scales, const uint32_t *a_offsets,
    const uint32_t *a_scales_offsets, const int32_t *expert_ids, int64_t total_tokens,
    int64_t scale_rows_total, int64_t I, int64_t K, int32_t num_experts,
    int32_t max_tokens_per_expert, int32_t num_active_experts, moeq_stream_t stream) {
    if (fmt != MOEQ_MXFP4 && fmt != MOEQ_MXFP8) return MOEQ_ERR_INVALID_ARG;
    if (I <= 0 || I % 128) return MOEQ_ERR_INVALID_ARG;
    moeq::GemmArgs ga;
    moeq_status st = blockscaled_common(fmt, 2, a, a_sf, b, b_sf, a_offsets, a_scales_offsets,
                                        expert_ids, total_tokens, scale_rows_total, 2 * I, K,
                                        num_experts, num_active_experts, &ga);
    if (st != MOEQ_OK) return st;
    if (expert_scales && !aligned16(expert_scales)) return MOEQ_ERR_INVALID_ARG;
    if (num_active_experts == 0 || total_tokens == 0) return MOEQ_OK;
    if (!c_q || !c_sf || !aligned16(c_q) || !aligned16(c_sf)) return MOEQ_ERR_INVALID_ARG;
    uint32_t *err = device_error_ptr();
    if (!err) return cuda_status(cudaErrorInvalidDevice);
    ga.expert_scales = expert_scales;
    ga.c_packed = c_q;
    ga.c_sf = c_sf;
    ga.max_tokens_per_expert = max_tokens_per_expert;
    ga.err = err;
    return cuda_status(moeq::launch_gemm(ga, stream));
}

}  // extern "C"
