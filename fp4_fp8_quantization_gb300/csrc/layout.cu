// Weight-preparation layout kernels: logical <-> tiled block-scale layout,
// and the gate/up row interleave of the fused SwiGLU GEMM's weight.
// ("max.nn.moe.NvMxf4f8Strategy", prepare_weight_scales: block scales
// rearranged into the kernel's layout.)  Byte shuffles, bound by HBM; run
// once per weight, off the per-step path.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moeq {

namespace {

// Byte (r, c) of a [rows, kv] logical scale matrix sits in the tiled buffer
// at atom (r / 128, c / 4) (atoms row-block-major, ceil(kv / 4) per row
// block), inner byte (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4.
__device__ __forceinline__ int64_t tiled_offset(int64_t r, int64_t c, int64_t kv_atoms) {
    return ((r >> 7) * kv_atoms + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// One thread per byte of the tiled output (padding bytes written as 0).
__global__ void sf_swizzle_kernel(uint8_t *__restrict__ tiled, const uint8_t *__restrict__ logical,
                                  int64_t batch, int64_t rows, int64_t kv) {
    pdl_wait();
    pdl_trigger();
    const int64_t kv_atoms = (kv + 3) / 4;
    const int64_t per_item = (rows + 127) / 128 * kv_atoms * 512;
    const int64_t total = batch * per_item;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / per_item, o = i - b * per_item;
        const int64_t atom = o >> 9, inner = o & 511;
        const int64_t rb = atom / kv_atoms, kb = atom - rb * kv_atoms;
        const int64_t r = rb * 128 + ((inner & 15) >> 2) * 32 + (inner >> 4);
        const int64_t c = kb * 4 + (inner & 3);
        tiled[i] = (r < rows && c < kv) ? logical[(b * rows + r) * kv + c] : (uint8_t)0;
    }
}

// One thread per logical byte.
__global__ void sf_unswizzle_kernel(uint8_t *__restrict__ logical,
                                    const uint8_t *__restrict__ tiled, int64_t batch,
                                    int64_t rows, int64_t kv) {
    pdl_wait();
    pdl_trigger();
    const int64_t kv_atoms = (kv + 3) / 4;
    const int64_t per_item = (rows + 127) / 128 * kv_atoms * 512;
    const int64_t total = batch * rows * kv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / (rows * kv), o = i - b * rows * kv;
        const int64_t r = o / kv, c = o - r * kv;
        logical[i] = tiled[b * per_item + tiled_offset(r, c, kv_atoms)];
    }
}

// out[b][2j] = gate[b][j], out[b][2j + 1] = up[b][j], rows of `words`
// 16-byte words (vec) or bytes.
template <typename T>
__global__ void interleave_rows_kernel(T *__restrict__ out, const T *__restrict__ gate,
                                       const T *__restrict__ up, int64_t batch, int64_t rows,
                                       int64_t words) {
    pdl_wait();
    pdl_trigger();
    const int64_t total = batch * rows * 2 * words;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t orow = i / words, w = i - orow * words;
        const int64_t b = orow / (2 * rows), jj = orow - b * 2 * rows;
        const int64_t src = (b * rows + (jj >> 1)) * words + w;
        out[i] = (jj & 1) ? up[src] : gate[src];
    }
}

int sm_count_cached() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    return cached_per_device(cache, dev, [dev]() {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    });
}

// grid-stride launches: up to 16 blocks of 256 threads per SM
int grid_for(int64_t n) {
    const int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)sm_count_cached() * 16;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_sf_swizzle(uint8_t *tiled, const uint8_t *logical, int64_t batch, int64_t rows,
                              int64_t kv, cudaStream_t s) {
    const int64_t n = batch * ((rows + 127) / 128) * ((kv + 3) / 4) * 512;
    if (n == 0) return cudaSuccess;
    return launch_pdl(sf_swizzle_kernel, grid_for(n), 256, 0, s, tiled, logical, batch, rows, kv);
}

cudaError_t launch_sf_unswizzle(uint8_t *logical, const uint8_t *tiled, int64_t batch,
                                int64_t rows, int64_t kv, cudaStream_t s) {
    const int64_t n = batch * rows * kv;
    if (n == 0) return cudaSuccess;
    return launch_pdl(sf_unswizzle_kernel, grid_for(n), 256, 0, s, logical, tiled, batch, rows,
                      kv);
}

cudaError_t launch_interleave_rows(uint8_t *out, const uint8_t *gate, const uint8_t *up,
                                   int64_t batch, int64_t rows, int64_t row_bytes,
                                   cudaStream_t s) {
    const int64_t n = batch * rows * 2 * row_bytes;
    if (n == 0) return cudaSuccess;
    const bool vec = row_bytes % 16 == 0 && ((uintptr_t)out | (uintptr_t)gate | (uintptr_t)up) % 16 == 0;
    if (vec)
        return launch_pdl(interleave_rows_kernel<uint4>, grid_for(n / 16), 256, 0, s,
                          reinterpret_cast<uint4 *>(out), reinterpret_cast<const uint4 *>(gate),
                          reinterpret_cast<const uint4 *>(up), batch, rows, row_bytes / 16);
    return launch_pdl(interleave_rows_kernel<uint8_t>, grid_for(n), 256, 0, s, out, gate, up,
                      batch, rows, row_bytes);
}

}  // namespace moeq
