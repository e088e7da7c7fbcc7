// Grouped (ragged mixture-of-experts) GEMMs on the 5th-generation tensor
// cores: FP8 rowwise-scaled, NVFP4 / MXFP4 / MXFP8 block-scaled, with a bf16
// epilogue or the fused SwiGLU + NVFP4 requantization epilogue.
//
// Pages: "grouped_matmul_rowwise_dynamic_scaled_fp8" (the rowwise formula,
// fp32 accumulation, scaled once after the reduction; its documented kernel is a
// naive one with no persistent or TMA path), "max.nn.moe.NvMxf4f8Strategy"
// (grouped_matmul: block-scaled with per-expert scales; grouped_matmul_swiglu:
// GEMM + SwiGLU + quantize in one kernel, byte-identical to the chained path).
//
// Design (persistent: one CTA per SM, or one CTA pair per two SMs):
//  * tile scheduler: every CTA builds, in shared memory, the prefix over
//    groups of ceil(rows_g / (128 * PAIR)) * (N / BN) tiles from the device
//    offsets, then walks tile ids cid, cid + (number of CTAs or pairs), ...;
//    a tile id maps to (group, m-block, n-block) by binary search on that
//    prefix, with n fastest so that concurrently running CTAs share A rows
//    and B[expert].
//  * FP4 kinds run M = 256 tiles over a CTA pair (cluster of two,
//    tcgen05 cta_group::2): each CTA stages its 128 A rows, half of the B
//    rows and all of the tile's B scales; the even CTA's thread issues the
//    MMAs for both; FP8 rowwise and MXFP8 run single-CTA 128-row tiles.
//  * warp 0 (one thread): TMA producer.  A tiles (128 rows x 128 bytes of K)
//    and B tiles land 128B-swizzled in a STAGES-deep shared-memory ring;
//    block-scaled kinds also load the 512-byte scale atoms of the k-tile
//    (contiguous in the tiled scale layout): tensor copies in pair tiles
//    (both B row blocks in one 3-D box), 1-D bulk copies otherwise.
//  * warp 1 (one thread): tcgen05.mma issuer.  The MMAs accumulate in TMEM
//    (FP8: two 128x256 accumulators, so the epilogue of tile i overlaps the
//    mainloop of tile i+1; block-scaled: one accumulator, because the
//    per-stage scale slots take the rest of TMEM); tcgen05.commit frees
//    ring stages and publishes finished accumulators.
//  * block-scaled kinds: two warps (one thread each) move each stage's
//    scale atoms shared -> TMEM with tcgen05.cp into that stage's TMEM slot
//    (the atoms dealt alternately) and signal the MMA thread through a
//    per-stage barrier, so the MMA thread issues only MMAs.
//  * remaining warps: epilogue.  Each warp owns a 32-lane quarter of TMEM
//    (one row per thread) and a column range; it reads 32 fp32 columns per
//    tcgen05.ld, frees the accumulator as soon as its columns are in
//    registers (single-accumulator kinds; in a pair with a relaxed arrive on
//    the even CTA's barrier), then applies the scales (and SwiGLU + the
//    requantization) in registers.
//  * every wait is bounded (about one second) and sets the device error
//    word instead of hanging.
#include <cstring>

#include "common.cuh"
#include "launch.h"

// Scale-load warp (1) or scale loads issued by the A/B producer (0).
#ifndef MOEQ_SF_LOADER
#define MOEQ_SF_LOADER 0
#endif

namespace moeq {

namespace {

enum Kind { kFp8Rowwise = 0, kNvfp4 = 1, kMxfp8 = 2, kMxfp4 = 3 };
// kSwiglu: SwiGLU + NVFP4 requant; kSwigluMx: SwiGLU + MX requant in the
// mainloop's element format (MXFP4 -> E2M1, MXFP8 -> E4M3, E8M0 scales).
enum Epi { kBf16 = 0, kSwiglu = 1, kSwigluMx = 2 };

// Groups a launch with the SiLU table may hold (its tile prefix shares the
// CTA's shared memory with the table).
constexpr int kSiluMaxGroups = 512;

template <int KIND, int EPI, int BN_, int STAGES_, int ACC_BUFS_, int EPI_WARPS_, int SF_WARPS_,
          int PAIR_, int SF_LOADER_ = 1, int SILU_TAB_ = 0>
struct Cfg {
    static constexpr int BM = 128;                              // rows of A per CTA
    static constexpr int PAIR = PAIR_;                          // CTAs per MMA (cta_group)
    static constexpr int MMA_M = BM * PAIR;
    static constexpr int BN = BN_;                              // columns of D per tile
    static constexpr int STAGES = STAGES_;
    static constexpr int ACC_BUFS = ACC_BUFS_;                  // TMEM accumulators
    static constexpr int BK_BYTES = 128;                        // one 128B swizzle row
    static constexpr int ELEMS_PER_BYTE = (KIND == kNvfp4 || KIND == kMxfp4) ? 2 : 1;
    static constexpr int BK = BK_BYTES * ELEMS_PER_BYTE;        // K elements per stage
    static constexpr int KSTEPS = 4;                            // 32 bytes of K per MMA
    static constexpr bool SCALED = KIND != kFp8Rowwise;
    static constexpr int SF_VEC = KIND == kNvfp4 ? 16 : 32;
    static constexpr int RB = BN >= 128 ? BN / 128 : 1;         // 128-row scale blocks of B
    static constexpr int SF_ATOMS = SCALED ? BK / SF_VEC / 4 : 0;   // atoms per 128 rows per stage
    static constexpr int SF_ATOM_BYTES = 512;
    static constexpr int B_ROWS_CTA = BN / PAIR;                // rows of B each CTA stages
    static constexpr int A_BYTES = BM * BK_BYTES;
    static constexpr int B_BYTES = B_ROWS_CTA * BK_BYTES;
    static constexpr int SFA_BYTES = SF_ATOMS * SF_ATOM_BYTES;
    // every CTA of a pair holds the scales of all BN rows of B: each CTA's
    // tensor cores produce all BN columns of its rows
    static constexpr int SFB_BYTES = SF_ATOMS * SF_ATOM_BYTES * RB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int EPI_WARPS = EPI_WARPS_;
    static constexpr int EPI_GROUPS = EPI_WARPS / 4;            // epilogue warps per TMEM quarter
    static constexpr int COLS_W = BN / EPI_GROUPS;              // accumulator columns per warp
    static constexpr int CHUNKS_W = COLS_W / 32;
    // warps issuing scale copies; 0: the MMA thread copies each stage's
    // scales right before its MMAs
    static constexpr int SF_WARPS = SCALED ? SF_WARPS_ : 0;
    static constexpr int SF_ITEMS = SF_ATOMS * (1 + RB);         // scale atoms per stage
    // 1: a warp of its own issues the scale loads, in parallel with the A/B
    // loads of warp 0
    static constexpr int SF_LOADER = SCALED ? SF_LOADER_ : 0;
    static constexpr int SF_WARP0 = 2 + SF_LOADER;
    static constexpr int EPI_WARP0 = SF_WARP0 + SF_WARPS;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    // SwiGLU epilogues: silu(gate) from a table of every bf16 gate in the
    // band where it has no closed form (32 KB, after the stages), where it
    // fits beside a tile prefix of kSiluMaxGroups groups; else computed
    static constexpr bool SILU_TAB =
        SILU_TAB_ && EPI != kBf16 &&
        STAGES * STAGE_BYTES + (int)kSiluTableBytes + 1024 + 4 * (kSiluMaxGroups + 1) + 512 <=
            227 * 1024;
    static constexpr int SILU_BYTES = SILU_TAB ? (int)kSiluTableBytes : 0;
    static constexpr int MAXG = SILU_TAB ? kSiluMaxGroups : kMaxGroups;  // groups per launch
    // fused SwiGLU epilogues on CTA pairs: the control warpgroups (producer,
    // MMA and scale-copy warps) give registers to the two epilogue
    // warpgroups (setmaxnreg acts per warpgroup and redistributes exactly the
    // registers the block is launched with; the host checks the compiled
    // count before launching).  Computing the SiLU (384 threads): control
    // 104, epilogue 200, without which the MX epilogue spills.  The table
    // kernels fit their 168 launch registers with 2 scale-copy warps; with 6
    // (512 threads, 128 at launch) the two control warpgroups keep 96 and the
    // epilogue gets 160.
    static constexpr int LAUNCH_REGS = 65536 / THREADS / 8 * 8;
    static constexpr bool NREG = EPI != kBf16 && PAIR_ == 2 && EPI_WARP0 % 4 == 0 &&
                                 EPI_WARPS == 8 && (SILU_TAB ? THREADS == 512 : THREADS == 384);
    static constexpr int NREG_CTRL = SILU_TAB ? 96 : 104;
    static constexpr int NREG_EPI =
        NREG ? (THREADS * LAUNCH_REGS - 32 * EPI_WARP0 * NREG_CTRL) / (32 * EPI_WARPS) / 8 * 8 : 0;
    static constexpr int ACC_COLS = BN;
    static constexpr int SF_COLS_A = SF_ATOMS * 4;
    static constexpr int SF_COLS_B = SF_ATOMS * 4 * RB;
    static constexpr int SF_COL0 = ACC_BUFS * ACC_COLS;
    static constexpr int SF_COLS_STAGE = SF_COLS_A + SF_COLS_B;
    static constexpr int TMEM_COLS = 512;
    // bf16 out: a 2 KB staging buffer per epilogue warp (one 32 x 32 chunk of
    // its rows) after the stages, for coalesced stores, where it fits (else
    // each thread stores its own row)
    static constexpr bool EPI_BUF_FITS =
        STAGES * STAGE_BYTES + EPI_WARPS * 2048 + 1024 <= 222 * 1024;
    static constexpr int EPI_BUF_BYTES = (EPI == kBf16 && EPI_BUF_FITS) ? 2048 : 0;
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + SILU_BYTES + 1024;
    static_assert(SF_COL0 + STAGES * SF_COLS_STAGE <= TMEM_COLS, "TMEM budget");
    static_assert(!NREG || (NREG_EPI >= LAUNCH_REGS && NREG_EPI <= 256 &&
                            32 * EPI_WARP0 * NREG_CTRL + 32 * EPI_WARPS * NREG_EPI <=
                                THREADS * LAUNCH_REGS),
                  "register split by warpgroups");
    // dynamic part + the tile prefix + the barriers and flags (under 512 bytes)
    static_assert(SMEM_BYTES + 4 * (MAXG + 1) + 512 <= 227 * 1024, "shared memory per CTA");
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
    static_assert(!SCALED || BN % 128 == 0, "block-scaled tiles cover whole 128-row scale atoms");
    static_assert(EPI_WARPS % 4 == 0 && COLS_W % 32 == 0 && COLS_W >= 32, "epilogue split");
    static_assert((ACC_BUFS == 2 && EPI == kBf16) || CHUNKS_W <= 4,
                  "single accumulator / SwiGLU epilogues drain TMEM to registers");
    static_assert(EPI != kSwigluMx || (CHUNKS_W % 2 == 0 && (KIND == kMxfp4 || KIND == kMxfp8)),
                  "an MX block is 64 accumulator columns of an MX mainloop");
    static_assert(ACC_BUFS == 1 || ACC_BUFS == 2, "accumulator buffers");
    static_assert(PAIR == 1 || (PAIR == 2 && BN == 256), "a pair splits a 256-row B tile in halves");
};

struct Params {
    const uint32_t *a_offsets;
    const uint32_t *a_sf_offsets;
    const int32_t *expert_ids;
    int num_groups, num_experts;
    int64_t total_rows, scale_rows_total;
    int N, K;
    const float *a_scales, *b_scales;
    const uint8_t *a_sf, *b_sf;
    const float *expert_scales;
    const float *out_tensor_scale;
    const uint16_t *row_scales;  // bf16 per row (SwiGLU + NVFP4), null = 1
    uint16_t *c;
    uint8_t *c_packed, *c_sf;
    uint32_t *err;
};

struct Tile {
    int g, mb, nb;
};

__device__ __forceinline__ Tile decode_tile(const uint32_t *prefix, int G, uint32_t t, int NB) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    uint32_t local = t - prefix[lo];
    Tile r;
    r.g = lo;
    r.mb = (int)(local / (uint32_t)NB);
    r.nb = (int)(local % (uint32_t)NB);
    return r;
}

// Tiles of group g (0 when the group is empty or its offsets / expert id /
// scale rows are unusable; those errors are reported by CTA 0 only).
template <class C, int EPI>
__device__ __forceinline__ uint32_t group_tiles(const Params &p, int g, int NB, bool report) {
    uint32_t r0 = __ldg(p.a_offsets + g), r1 = __ldg(p.a_offsets + g + 1);
    int e = __ldg(p.expert_ids + g);
    if (r1 < r0 || (int64_t)r1 > p.total_rows) {
        if (report) set_error(p.err, MOEQ_DEVERR_BAD_OFFSETS);
        return 0;
    }
    if (e < 0 || e >= p.num_experts) {
        if (report) set_error(p.err, MOEQ_DEVERR_BAD_EXPERT);
        return 0;
    }
    uint32_t rows = r1 - r0;
    if (C::SCALED || EPI != kBf16) {
        uint32_t s0 = __ldg(p.a_sf_offsets + g), s1 = __ldg(p.a_sf_offsets + g + 1);
        uint32_t need = (rows + 127u) & ~127u;
        if ((s0 & 127u) || s1 < s0 || s1 - s0 < need || (int64_t)s1 > p.scale_rows_total) {
            if (report) set_error(p.err, MOEQ_DEVERR_SCALE_ROWS);
            return 0;
        }
    }
    // a CTA pair takes two consecutive m-blocks of the group
    return ((rows + C::BM - 1) / C::BM + C::PAIR - 1) / C::PAIR * (uint32_t)NB;
}

__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z),
                 "r"(w)
                 : "memory");
}

// TMA tensor store of a shared-memory box (bulk async-group of this thread)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     map),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the thread's bulk stores have read their shared memory / have completed
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}


__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

// Epilogue of one 32-column accumulator chunk of this thread's row.
//   bf16 out: c[row, n] = bf16(acc * scale(s)); FP8 rowwise applies
//             a_scale (rs) then b_scale[e, n]; block-scaled the expert scale.
//             With a staging buffer, the warp's 32 x 32 chunk is written into
//             it (sbuf, a shared address; 64-byte rows whose 16-byte pieces
//             are XOR-swizzled by row pair: the tensor map's 64-byte swizzle,
//             free of bank conflicts) and leaves as one tensor store (tmc)
//             when all 32 rows lie in the group; otherwise it is read back
//             transposed and stored with four lanes per row, 8 rows of 64
//             contiguous bytes per instruction, the warp's first nvalid rows
//             only.  Without a buffer, each valid thread stores its row.
//   SwiGLU:   16 (gate, up) pairs -> 16 h -> one NVFP4 block; returns the
//             E4M3 scale code, writes the 8 packed bytes.  gate and up are
//             bf16((acc * s) * rsr): s the expert scale, rsr the row scale
//             (1 without row scales, an exact no-op).
// h = silu(gate) * up for two (gate, up) pairs of bf16 values held in fp32
// (gates in the low halves of q0, q1, ups in the high halves): silu from
// the table at shared-memory address stab, which holds exactly the computed
// values and reduces to the same closed forms outside its band, or computed.
template <bool TAB>
__device__ __forceinline__ F2 swiglu_pairs(F2 q0, F2 q1, uint32_t stab) {
    if constexpr (TAB)
        return mul2(f2(silu_lookup_shared(__float_as_uint(f2_lo(q0)) >> 16, stab),
                       silu_lookup_shared(__float_as_uint(f2_lo(q1)) >> 16, stab)),
                    f2(f2_hi(q0), f2_hi(q1)));
    else
        return swiglu2(f2_lo(q0), f2_lo(q1), f2_hi(q0), f2_hi(q1));
}

template <class C, int KIND, int EPI>
__device__ __forceinline__ uint32_t epilogue_chunk(const Params &p, const uint32_t (&r)[32],
                                                   int nc, int e, int64_t row, bool valid,
                                                   float rs, float inv_out, float rsr = 1.0f,
                                                   uint32_t sbuf = 0, int nvalid = 0,
                                                   const CUtensorMap *tmc = nullptr,
                                                   uint32_t stab = 0) {
    if (EPI == kBf16) {
        const int lane = threadIdx.x & 31;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = nc + j * 8;
            float bs[8];
            if (KIND == kFp8Rowwise) {
#pragma unroll
                for (int i = 0; i < 8; ++i) bs[i] = 0.0f;
                if (n < p.N) {  // N is a multiple of 16: n + 8 <= N
                    const float4 *bp =
                        reinterpret_cast<const float4 *>(p.b_scales + (int64_t)e * p.N + n);
                    float4 b0 = __ldg(bp), b1 = __ldg(bp + 1);
                    bs[0] = b0.x; bs[1] = b0.y; bs[2] = b0.z; bs[3] = b0.w;
                    bs[4] = b1.x; bs[5] = b1.y; bs[6] = b1.z; bs[7] = b1.w;
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float v0 = __uint_as_float(r[j * 8 + 2 * i]);
                float v1 = __uint_as_float(r[j * 8 + 2 * i + 1]);
                if (KIND == kFp8Rowwise) {
                    v0 = __fmul_rn(__fmul_rn(v0, rs), bs[2 * i]);
                    v1 = __fmul_rn(__fmul_rn(v1, rs), bs[2 * i + 1]);
                } else {
                    v0 = __fmul_rn(v0, rs);
                    v1 = __fmul_rn(v1, rs);
                }
                w[j * 4 + i] = f32_to_bf16_bits(v0) | (f32_to_bf16_bits(v1) << 16);
            }
        }
        if (C::EPI_BUF_BYTES == 0) {
            if (valid) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = nc + j * 8;
                    if (n < p.N && store_ok(row < p.total_rows && n + 8 <= p.N, p.err))
                        st_global_v4(p.c + row * p.N + n, w[j * 4], w[j * 4 + 1], w[j * 4 + 2],
                                     w[j * 4 + 3]);
                }
            }
            return 0u;
        }
        if (nc >= p.N) return 0u;  // a chunk past N (N a multiple of 16, not of 32)
        // the previous chunk's reads of the buffer are done (the lanes' and
        // the tensor store's)
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_shared_v4(sbuf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), w[j * 4],
                         w[j * 4 + 1], w[j * 4 + 2], w[j * 4 + 3]);
        if (nvalid == 32) {
            // a whole 32-row chunk: one tensor store (the buffer's layout is
            // the 64-byte swizzle of the tensor map; columns past N and rows
            // past the output are clipped by the copy)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(tmc, sbuf, nc, (int)(row - lane));
                bulk_commit();
            }
            return 0u;
        }
        __syncwarp();
        const int k = lane & 3;
        const int n = nc + k * 8;
        const int64_t row0 = row - lane;  // the warp's first row
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = (lane >> 2) + 8 * i;
            const uint4 v = ld_shared_v4(sbuf + rr * 64 + ((k ^ ((rr >> 1) & 3)) << 4));
            if (rr < nvalid && n < p.N &&
                store_ok(row0 + rr < p.total_rows && n + 8 <= p.N, p.err))
                st_global_v4(p.c + (row0 + rr) * p.N + n, v.x, v.y, v.z, v.w);
        }
        return 0u;
    } else {
        // h = silu(gate) * up with gate, up = bf16(acc * scale), in paired
        // fp32 arithmetic (bit-identical to the scalar definition)
        float h[16];
        const F2 rs2 = f2(rs, rs), rr2 = f2(rsr, rsr);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const F2 q0 = round_bf16_2(mul2(
                mul2(f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), rs2), rr2));
            const F2 q1 = round_bf16_2(mul2(
                mul2(f2(__uint_as_float(r[2 * i + 2]), __uint_as_float(r[2 * i + 3])), rs2), rr2));
            const F2 hh = swiglu_pairs<C::SILU_TAB>(q0, q1, stab);
            h[i] = f2_lo(hh);
            h[i + 1] = f2_hi(hh);
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(h[i]));
        const Nvfp4Scale s = nvfp4_block_scale(m, inv_out);
        float lo8[8], hi8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo8[i] = h[i];
            hi8[i] = h[8 + i];
        }
        const uint32_t c0 = nvfp4_codes8(lo8, s.r);
        const uint32_t c1 = nvfp4_codes8(hi8, s.r);
        if (valid && store_ok(row < p.total_rows && nc / 4 + 8 <= p.N / 4, p.err))
            *reinterpret_cast<uint2 *>(p.c_packed + row * (p.N / 4) + nc / 4) = make_uint2(c0, c1);
        return s.code;
    }
}

// Bytes one CTA's loading warp l issues per stage in pair tiles (warp 0:
// the A and B tiles, and the scale atoms too without a scale loader; the
// scale loader: the A and all B scale atoms).
template <class C>
__device__ __forceinline__ uint32_t loader_bytes(int l) {
    const uint32_t ab = C::A_BYTES + C::B_BYTES;
    const uint32_t sf = C::SCALED ? C::SFA_BYTES + C::RB * C::SF_ATOMS * C::SF_ATOM_BYTES : 0u;
    return C::SF_LOADER ? (l == 0 ? ab : sf) : ab + sf;
}

// Stores the NVFP4 scale bytes of `nblk` consecutive blocks (nblk = 1, 2 or
// 4 chunks of 32 accumulator columns) starting at accumulator column nc0.
__device__ __forceinline__ void store_sf_bytes(const Params &p, int64_t prow, int nc0,
                                               uint32_t bytes, int nblk) {
    const int64_t kv_atoms = p.N / 128;
    const int blk = nc0 / 32;  // first NVFP4 block of the output row
    if (!store_ok(prow < p.scale_rows_total && blk + nblk <= p.N / 32, p.err)) return;
    uint8_t *w = p.c_sf + sf_word_offset(prow, blk / 4, kv_atoms) + (blk & 3);
    if (nblk == 4)
        *reinterpret_cast<uint32_t *>(w) = bytes;
    else if (nblk == 2)
        *reinterpret_cast<uint16_t *>(w) = (uint16_t)bytes;
    else
        *w = (uint8_t)bytes;
}

// Copies the scale atoms of one stage shared -> TMEM (the atoms with index
// j % nw == w).  A atom ks -> columns 4 ks of the stage's slot; B atom
// (rb, ks) -> columns 4 (ks RB + rb), so each MMA step reads 4 RB
// consecutive columns covering its BN rows.  In a CTA pair the copy writes
// each CTA's tensor memory from its own shared memory.
template <class C>
__device__ __forceinline__ void copy_stage_scales(uint32_t tmem, const uint8_t *smem, int stage,
                                                  int w, int nw) {
    const uint32_t ssfa = smem_u32(smem + stage * C::STAGE_BYTES) + C::A_BYTES + C::B_BYTES;
    const uint32_t ssfb = ssfa + C::SFA_BYTES;
    const uint32_t tsfa = tmem + C::SF_COL0 + stage * C::SF_COLS_STAGE;
    const uint32_t tsfb = tsfa + C::SF_COLS_A;
#pragma unroll
    for (int j = 0; j < C::SF_ITEMS; ++j) {
        if (j % nw != w) continue;
        if (j < C::SF_ATOMS) {
            tmem_cp_sf_atom<C::PAIR>(tsfa + 4 * j, sdesc_sf_atom(ssfa + 512 * j));
        } else {
            const int i = (j - C::SF_ATOMS) / C::RB, rb = (j - C::SF_ATOMS) % C::RB;
            tmem_cp_sf_atom<C::PAIR>(tsfb + 4 * (i * C::RB + rb),
                                     sdesc_sf_atom(ssfb + 512 * (rb * C::SF_ATOMS + i)));
        }
    }
}

// SwiGLU + MX requant of 64 accumulator columns (32 (gate, up) pairs, one
// 32-element MX block) of this thread's row: h as in the NVFP4 epilogue
// (gate, up = bf16(acc * s)), then the MX rule of the quantizer on the fp32
// h (scale code from the block amax, elements = elem(h * 2^(127 - c))).
// Writes 32 (E4M3) or 16 (packed E2M1) bytes; returns the E8M0 code.
template <int KIND, bool TAB>
__device__ __forceinline__ uint32_t epilogue_mx_block(const Params &p, const uint32_t (&r0)[32],
                                                      const uint32_t (&r1)[32], int nc,
                                                      int64_t row, bool valid, float rs,
                                                      uint32_t stab) {
    float h[32];
    const F2 rs2 = f2(rs, rs);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint32_t(&r)[32] = half ? r1 : r0;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const F2 q0 = round_bf16_2(
                mul2(f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), rs2));
            const F2 q1 = round_bf16_2(
                mul2(f2(__uint_as_float(r[2 * i + 2]), __uint_as_float(r[2 * i + 3])), rs2));
            const F2 hh = swiglu_pairs<TAB>(q0, q1, stab);
            h[half * 16 + i] = f2_lo(hh);
            h[half * 16 + i + 1] = f2_hi(hh);
        }
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(h[i]));
    uint32_t code = 0;
    float f = 0.0f;
    if (m != 0.0f) {
        code = mx_scale_code_f32(m, KIND == kMxfp8 ? 8 : 2);
        f = mx_multiplier(code);
    }
    const F2 f2v = f2(f, f);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const F2 t = mul2(f2(h[i], h[i + 1]), f2v);
        h[i] = f2_lo(t);
        h[i + 1] = f2_hi(t);
    }
    if (valid) {
        if (KIND == kMxfp8) {
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                w[j] = m == 0.0f ? 0u
                                 : (e4m3x2(h[4 * j], h[4 * j + 1]) |
                                    (e4m3x2(h[4 * j + 2], h[4 * j + 3]) << 16));
            uint8_t *o = p.c_packed + row * (p.N / 2) + nc / 2;
            if (store_ok(row < p.total_rows && nc / 2 + 32 <= p.N / 2, p.err)) {
                st_global_v4(o, w[0], w[1], w[2], w[3]);
                st_global_v4(o + 16, w[4], w[5], w[6], w[7]);
            }
        } else {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float x8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) x8[i] = h[8 * j + i];
                w[j] = m == 0.0f ? 0u : e2m1x8(x8);
            }
            if (store_ok(row < p.total_rows && nc / 4 + 16 <= p.N / 4, p.err))
                st_global_v4(p.c_packed + row * (p.N / 4) + nc / 4, w[0], w[1], w[2], w[3]);
        }
    }
    return code;
}

// Stores the E8M0 scale byte of the MX block starting at accumulator column
// nc (output element nc / 2, block nc / 64) of logical scale row prow.
__device__ __forceinline__ void store_sf_byte_mx(const Params &p, int64_t prow, int nc,
                                                 uint32_t code) {
    const int64_t kv_atoms = (p.N / 64 + 3) / 4;
    const int blk = nc / 64;
    if (store_ok(prow < p.scale_rows_total && blk < p.N / 64, p.err))
        p.c_sf[sf_word_offset(prow, blk / 4, kv_atoms) + (blk & 3)] = (uint8_t)code;
}

template <class C, int KIND, int EPI>
__global__ void __launch_bounds__(C::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA,
                        const __grid_constant__ CUtensorMap tmSFB,
                        const __grid_constant__ CUtensorMap tmC, const Params p) {
    constexpr bool PAIRED = C::PAIR > 1;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full_bar[C::STAGES];
    __shared__ uint64_t empty_bar[C::STAGES];
    __shared__ uint64_t tfull_bar[C::ACC_BUFS];
    __shared__ uint64_t tempty_bar[C::ACC_BUFS];
    __shared__ uint64_t drain_bar;
    __shared__ uint64_t sf_bar[C::STAGES];     // scale atoms of a stage are in TMEM
    __shared__ uint64_t sf_drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ uint32_t prefix[C::MAXG + 1];
    // stages each loading warp of this CTA went through (announced on the
    // barrier, copies issued), stored once when it stops; read by the even
    // CTA at teardown
    constexpr int LOADERS = 1 + C::SF_LOADER;
    __shared__ uint32_t stages_done[LOADERS];

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.num_groups;
    const int NB = (p.N + C::BN - 1) / C::BN;
    volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) {
            // one arrival per loading warp (in a pair, the even CTA's
            // loaders announce the bytes of both CTAs)
            mbar_init(&full_bar[s], LOADERS);
            mbar_init(&empty_bar[s], 1);
        }
#pragma unroll
        for (int l = 0; l < LOADERS; ++l) stages_done[l] = 0;
#pragma unroll
        for (int b = 0; b < C::ACC_BUFS; ++b) {
            mbar_init(&tfull_bar[b], 1);
            // the even CTA's MMA thread waits for the epilogues of both CTAs
            mbar_init(&tempty_bar[b], C::PAIR * C::EPI_WARPS);
        }
        mbar_init(&drain_bar, 1);
        mbar_init(&sf_drain_bar, C::SF_WARPS > 0 ? C::SF_WARPS : 1);  // one commit per scale warp
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&sf_bar[s], C::SF_WARPS > 0 ? C::SF_WARPS : 1);
        abort_flag = 0;
        prefix[0] = 0;
        fence_barrier_init();
    }
    // the SiLU table, after the stages (visible after the barrier below)
    constexpr int kSiluOff = C::STAGES * C::STAGE_BYTES + C::EPI_WARPS * C::EPI_BUF_BYTES;
    if constexpr (C::SILU_TAB) build_silu_table(reinterpret_cast<float *>(smem + kSiluOff));
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (PAIRED && C::SCALED) {
            prefetch_tensormap(&tmSFA);
            prefetch_tensormap(&tmSFB);
        }
    }
    // everything above touches only shared memory and the kernel parameters;
    // from here on global memory written by the preceding kernel is read
    pdl_wait();
    if (warp == 1) {  // in a pair, warp 1 of both CTAs allocates collectively
        tmem_alloc<C::PAIR>(&tmem_slot, C::TMEM_COLS);
        tmem_relinquish<C::PAIR>();
    }
    for (int g = threadIdx.x; g < G; g += blockDim.x)
        prefix[g + 1] = group_tiles<C, EPI>(p, g, NB, blockIdx.x == 0);
    __syncthreads();
    if (warp == 0) {  // inclusive prefix over prefix[1..G]
        uint32_t carry = 0;
        for (int base = 0; base < G; base += 32) {
            int g = base + lane;
            uint32_t v = g < G ? prefix[g + 1] : 0u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
                if (lane >= o) v += t;
            }
            if (g < G) prefix[g + 1] = carry + v;
            carry += __shfl_sync(0xFFFFFFFFu, v, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // a pair: the other CTA's barriers must be initialised before any copy,
    // commit or arrival targets them
    if (PAIRED) cluster_sync();
    const uint32_t total = prefix[G];
    const uint32_t tmem = tmem_slot;
    const int KT = p.K / C::BK;
    const uint32_t rank = PAIRED ? cluster_ctarank() : 0u;   // m-block within the pair
    const uint32_t cid = blockIdx.x / C::PAIR, ncl = gridDim.x / C::PAIR;

    if (warp < C::EPI_WARP0) {
    if constexpr (C::NREG) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::NREG_CTRL));
    if (warp == 0 || (C::SF_LOADER && warp == 2)) {
        // ------------------------------------------------ TMA producers
        // Warp 0 loads the A and B tiles, warp 2 (or warp 0 as well, without
        // a scale loader) the scale atoms; each arrives on the stage's full
        // barrier with its byte count and counts the stages it went through.
        // Both CTAs of a pair load their own A rows, their half of the B
        // rows and all of the tile's scales; the copies of both complete on
        // the even CTA's full barrier, whose loaders expect the bytes of
        // both CTAs (the odd CTA's loaders only issue).
        const bool do_ab = warp == 0;
        const bool do_sf = C::SCALED && (warp == 2 || !C::SF_LOADER);
        const int loader = warp == 0 ? 0 : 1;
        if (lane == 0) {
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b = policy_evict_last();
            const int64_t kv_atoms = C::SCALED ? (int64_t)p.K / C::SF_VEC / 4 : 0;
            const int nrb = (p.N + 127) / 128;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t visits = 0;
            bool ok = true;
            for (uint32_t t = cid; ok && t < total; t += ncl) {
                const Tile tl = decode_tile(prefix, G, t, NB);
                const int mb = tl.mb * C::PAIR + (int)rank;
                const int e = __ldg(p.expert_ids + tl.g);
                const int row0 = (int)__ldg(p.a_offsets + tl.g) + mb * C::BM;
                const int n0 = tl.nb * C::BN;
                int64_t sfa0 = 0, sfb0 = 0;
                int rbs = 1;  // scale row-blocks of B present in this tile
                if (C::SCALED) {
                    // an m-block past the group's end (the odd CTA of a pair
                    // on a group with an odd m-block count) computes
                    // discarded rows: point its A scales at a real m-block so
                    // the copy stays inside the scale buffer
                    const uint32_t rgp = __ldg(p.a_offsets + tl.g + 1) - __ldg(p.a_offsets + tl.g);
                    const int mlast = (int)((rgp + C::BM - 1) / C::BM) - 1;
                    sfa0 = ((int64_t)(__ldg(p.a_sf_offsets + tl.g) >> 7) + min(mb, mlast)) * kv_atoms;
                    sfb0 = ((int64_t)e * nrb + n0 / 128) * kv_atoms;
                    rbs = min(C::RB, nrb - n0 / 128);
                }
                if (PAIRED) rbs = C::RB;  // one box of RB row blocks (see below)
                const uint32_t tx =
                    (do_ab ? (uint32_t)(C::A_BYTES + C::B_BYTES) : 0u) +
                    (do_sf ? (uint32_t)(C::SFA_BYTES + rbs * C::SF_ATOMS * C::SF_ATOM_BYTES) : 0u);
                for (int kt = 0; kt < KT; ++kt) {
                    if (!mbar_wait<PAIRED>(&empty_bar[stage], phase ^ 1u, abort_v, p.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * C::STAGE_BYTES;
                    uint8_t *sb = sa + C::A_BYTES;
                    uint8_t *ssfa = sb + C::B_BYTES;
                    uint8_t *ssfb = ssfa + C::SFA_BYTES;
                    bool stuck = false;
#ifdef MOEQ_TEST_STUCK_STAGE
                    // failure-detection test build: the first stage of the
                    // CTA's first tile is announced but never loaded, so every
                    // wait on it runs into its time limit
                    stuck = t == cid && kt == 0;
#endif
                    ++visits;
                    if (!PAIRED) {
                        mbar_arrive_expect_tx(&full_bar[stage], tx);
                        if (do_ab && !stuck) {
                            tma_load_2d(sa, &tmA, &full_bar[stage], kt * C::BK_BYTES, row0, pol_a);
                            tma_load_3d(sb, &tmB, &full_bar[stage], kt * C::BK_BYTES, n0, e, pol_b);
                        }
                        if (do_sf && !stuck) {
                            bulk_load(ssfa, p.a_sf + (sfa0 + (int64_t)kt * C::SF_ATOMS) * 512,
                                      C::SFA_BYTES, &full_bar[stage]);
                            for (int rb = 0; rb < rbs; ++rb)
                                bulk_load(ssfb + rb * C::SF_ATOMS * 512,
                                          p.b_sf + (sfb0 + rb * kv_atoms + (int64_t)kt * C::SF_ATOMS) * 512,
                                          C::SF_ATOMS * 512, &full_bar[stage]);
                        }
                    } else {
                        const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
                        if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2u * tx);
                        if (do_ab && !stuck) {
                            tma_load_2d_pair(sa, &tmA, fb, kt * C::BK_BYTES, row0, pol_a);
                            tma_load_3d_pair(sb, &tmB, fb, kt * C::BK_BYTES,
                                             n0 + (int)rank * C::B_ROWS_CTA, e, pol_b);
                        }
                        if (do_sf && !stuck) {
                            // scale buffers viewed as rows of 256 bytes: an
                            // atom is two rows
                            tma_load_2d_pair(ssfa, &tmSFA, fb, 0,
                                             (int)((sfa0 + (int64_t)kt * C::SF_ATOMS) * 2), pol_a);
                            // all RB row blocks of B scales in one copy (a row
                            // block past the expert's N reads the next
                            // expert's or zero-filled rows, never used)
                            tma_load_3d_pair(ssfb, &tmSFB, fb, 0, kt * C::SF_ATOMS * 2,
                                             e * nrb + n0 / 128, pol_b);
                        }
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            stages_done[loader] = visits;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // (the even CTA of a pair issues the MMAs of both)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t t = cid; ok && t < total; t += ncl, ++it) {
                const uint32_t buf = C::ACC_BUFS == 2 ? (it & 1u) : 0u;
                const uint32_t aph = C::ACC_BUFS == 2 ? ((it >> 1) & 1u) : (it & 1u);
                if (!mbar_wait<PAIRED>(&tempty_bar[buf], aph ^ 1u, abort_v, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * C::ACC_COLS;
                for (int kt = 0; kt < KT; ++kt) {
                    // with scale warps, they signal once the stage's operands
                    // have landed and its scales are in TMEM
                    const bool waited = C::SF_WARPS
                                            ? mbar_wait(&sf_bar[stage], phase, abort_v, p.err)
                                            : mbar_wait<PAIRED>(&full_bar[stage], phase, abort_v,
                                                                p.err);
                    if (!waited) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (C::SCALED && C::SF_WARPS == 0) copy_stage_scales<C>(tmem, smem, stage, 0, 1);
                    const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + C::A_BYTES;
                    const uint32_t tsfa = tmem + C::SF_COL0 + stage * C::SF_COLS_STAGE;
                    const uint32_t tsfb = tsfa + C::SF_COLS_A;
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS; ++ks) {
                        const uint64_t ad = sdesc_sw128(sa + ks * 32);
                        const uint64_t bd = sdesc_sw128(sb + ks * 32);
                        const uint32_t acc = (kt | ks) ? 1u : 0u;
                        if (KIND == kFp8Rowwise) {
                            mma_f8f6f4<C::PAIR>(d, ad, bd, idesc_f8_e4m3(C::MMA_M, C::BN), acc);
                        } else if (KIND == kNvfp4) {
                            mma_nvf4<C::PAIR>(d, ad, bd, idesc_nvf4(C::MMA_M, C::BN), tsfa + 4 * ks,
                                              tsfb + 4 * C::RB * ks, acc);
                        } else if (KIND == kMxfp4) {
                            // scale atom ks / 2 holds 4 blocks of 32 = two K=64 steps
                            mma_mxf4<C::PAIR>(d, ad, bd, idesc_mxf4(C::MMA_M, C::BN, (ks & 1) * 2),
                                              tsfa + 4 * (ks >> 1), tsfb + 4 * C::RB * (ks >> 1),
                                              acc);
                        } else {
                            mma_mxf8<C::PAIR>(d, ad, bd, idesc_mxf8_e4m3(C::MMA_M, C::BN, ks), tsfa,
                                              tsfb, acc);
                        }
                    }
                    // the stage is free in both CTAs once these MMAs are done
                    if (!PAIRED)
                        tc_commit(&empty_bar[stage]);
                    else
                        tc_commit_mc<2>(&empty_bar[stage], 0x3);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    if (!PAIRED)
                        tc_commit(&tfull_bar[buf]);
                    else
                        tc_commit_mc<2>(&tfull_bar[buf], 0x3);
                }
            }
            // every tcgen05 operation issued here completes before TMEM is freed
            tc_commit<C::PAIR>(&drain_bar);
            mbar_drain(&drain_bar, 0);
        }
    } else if (C::SF_WARPS && warp >= C::SF_WARP0 && warp < C::EPI_WARP0) {
        // ------------------------------------------------ scale copies
        // Copies each stage's scale atoms shared -> TMEM (tcgen05.cp) ahead of
        // the MMA thread and publishes them with tcgen05.commit on sf_bar.
        // A stage's TMEM scale slot is rewritten only after full_bar of its
        // next use, which the producer can only reach after the MMAs that
        // read the slot have completed (empty_bar), so the slot is free.
        const int sfw = warp - C::SF_WARP0;
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (uint32_t t = cid; t < total; t += ncl) {
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!mbar_wait<PAIRED>(&full_bar[stage], phase, abort_v, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    copy_stage_scales<C>(tmem, smem, stage, sfw, C::SF_WARPS);
                    tc_commit<C::PAIR>(&sf_bar[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            tc_commit<C::PAIR>(&sf_drain_bar);
            mbar_drain(&sf_drain_bar, 0);
        }
    }
    } else {
    if constexpr (C::NREG) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::NREG_EPI));
    {
        // ------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int cgrp = (warp - C::EPI_WARP0) >> 2;  // column group of this warp
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // accumulator release: on the even CTA's barrier
        const uint32_t tempty0 = PAIRED ? mapa_shared(smem_u32(&tempty_bar[0]), 0) : 0u;
        auto release = [&](uint32_t buf) {
            if (!PAIRED)
                mbar_arrive(&tempty_bar[buf]);
            else
                mbar_arrive_cluster_relaxed(tempty0 + 8u * buf);
        };
        const uint32_t silu_tab = smem_u32(smem + kSiluOff);
        // this warp's bf16 staging buffer, after the stages
        const uint32_t sbuf = smem_u32(smem + C::STAGES * C::STAGE_BYTES) +
                              (uint32_t)(warp - C::EPI_WARP0) * C::EPI_BUF_BYTES;
        uint32_t it = 0;
        for (uint32_t t = cid; t < total; t += ncl, ++it) {
            const uint32_t buf = C::ACC_BUFS == 2 ? (it & 1u) : 0u;
            const uint32_t aph = C::ACC_BUFS == 2 ? ((it >> 1) & 1u) : (it & 1u);
            const Tile tl = decode_tile(prefix, G, t, NB);
            const int e = __ldg(p.expert_ids + tl.g);
            const uint32_t r0 = __ldg(p.a_offsets + tl.g);
            const uint32_t rg = __ldg(p.a_offsets + tl.g + 1) - r0;
            const int mb = tl.mb * C::PAIR + (int)rank;
            // scale rows of this m-block exist only if the group reaches it
            const bool mb_in_group = (uint32_t)mb * C::BM < rg;
            const uint32_t lrow = (uint32_t)(mb * C::BM + quad * 32 + lane);
            const bool valid = lrow < rg;
            const int64_t row = (int64_t)r0 + lrow;
            const int ncol0 = tl.nb * C::BN + cgrp * C::COLS_W;
            // rows of this warp's 32 that lie in the group
            const int64_t left = (int64_t)rg - (int64_t)(mb * C::BM + quad * 32);
            const int nvalid = left <= 0 ? 0 : (left >= 32 ? 32 : (int)left);
            float rs = 1.0f, inv_out = 0.0f;
            if (KIND == kFp8Rowwise) {
                rs = valid ? __ldg(p.a_scales + row) : 0.0f;
            } else if (p.expert_scales) {
                rs = __ldg(p.expert_scales + e);
            }
            if (EPI == kSwiglu) inv_out = __fdiv_rn(1.0f, __ldg(p.out_tensor_scale + e));
            const float rsr = (EPI == kSwiglu && p.row_scales && valid)
                                  ? bf16_bits_to_f32(__ldg(p.row_scales + row))
                                  : 1.0f;
            if (!mbar_wait<PAIRED>(&tfull_bar[buf], aph, abort_v, p.err)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + lane_off + buf * C::ACC_COLS + cgrp * C::COLS_W;
            uint32_t sfbytes = 0;
            if (ncol0 >= p.N) {
                // this warp's columns lie past N (last n-block of an N that is
                // not a multiple of BN): nothing to read or write
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release(buf);
                continue;
            }
            if (C::ACC_BUFS == 1 || EPI != kBf16) {
                // drain this warp's columns to registers, free TMEM, then compute
                uint32_t r[C::CHUNKS_W > 4 ? 4 : C::CHUNKS_W][32];
#pragma unroll
                for (int ch = 0; ch < (C::CHUNKS_W > 4 ? 4 : C::CHUNKS_W); ++ch)
                    tmem_ld32(tbase + ch * 32, r[ch]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release(buf);
                if (EPI == kSwigluMx) {
                    const int64_t prow = (int64_t)__ldg(p.a_sf_offsets + tl.g) + lrow;
#pragma unroll
                    for (int b2 = 0; b2 < (C::CHUNKS_W > 4 ? 4 : C::CHUNKS_W) / 2; ++b2) {
                        const uint32_t code = epilogue_mx_block<KIND, C::SILU_TAB>(
                            p, r[2 * b2], r[2 * b2 + 1], ncol0 + b2 * 64, row, valid, rs,
                            silu_tab);
                        if (mb_in_group) store_sf_byte_mx(p, prow, ncol0 + b2 * 64, valid ? code : 0u);
                    }
                } else {
#pragma unroll
                    for (int ch = 0; ch < (C::CHUNKS_W > 4 ? 4 : C::CHUNKS_W); ++ch)
                        sfbytes |= epilogue_chunk<C, KIND, EPI>(p, r[ch], ncol0 + ch * 32, e, row,
                                                                valid, rs, inv_out, rsr, sbuf,
                                                                nvalid, &tmC, silu_tab)
                                   << (8 * ch);
                }
            } else {
#pragma unroll 1
                for (int ch = 0; ch < C::CHUNKS_W; ++ch) {
                    uint32_t r[32];
                    tmem_ld32(tbase + ch * 32, r);
                    tmem_ld_wait();
                    if (ch == C::CHUNKS_W - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) release(buf);
                    }
                    epilogue_chunk<C, KIND, EPI>(p, r, ncol0 + ch * 32, e, row, valid, rs,
                                                 inv_out, 1.0f, sbuf, nvalid, &tmC);
                }
            }
            if (EPI == kSwiglu && mb_in_group) {
                const int nblk = C::CHUNKS_W < 4 ? C::CHUNKS_W : 4;
                store_sf_bytes(p, (int64_t)__ldg(p.a_sf_offsets + tl.g) + lrow, ncol0,
                               valid ? sfbytes : 0u, nblk);
            }
        }
        // this warp's tensor stores have completed
        if (C::EPI_BUF_BYTES && lane == 0) bulk_wait_all();
    }
    }

    // this CTA's loads, MMAs and stores are all issued: the next kernel's
    // CTAs may launch (they wait for this grid's completion before touching
    // memory)
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    // every loader of both CTAs has stopped issuing
    if (PAIRED) cluster_sync();
    if (threadIdx.x == 0 && rank == 0) {
        // Every issued copy lands before either CTA may leave, after an
        // abort too.  No loader of either CTA reaches phase p + 1 of a stage
        // before every loader reached phase p (it first waits for the MMAs
        // that consumed phase p), so the counts differ by at most one and
        // only the current phase n - 1 of a stage can be incomplete.  For it,
        // each loader l of the even CTA that did not arrive arrives now,
        // expecting the bytes of its odd-CTA counterpart if that one issued
        // them; if the even loader arrived (expecting both CTAs' bytes) but
        // its odd counterpart issued nothing, those bytes are completed
        // here; then the phase is waited for with a bound.
        uint32_t v0[LOADERS], v1[LOADERS];
#pragma unroll
        for (int l = 0; l < LOADERS; ++l) {
            v0[l] = stages_done[l];
            v1[l] = PAIRED ? ld_cluster_u32(mapa_shared(smem_u32(&stages_done[l]), 1)) : v0[l];
        }
        // phases of stage s a loader went through after v stages in all
        auto phases = [](uint32_t v, int s) {
            return v / C::STAGES + ((uint32_t)s < v % C::STAGES ? 1u : 0u);
        };
        for (int s = 0; s < C::STAGES; ++s) {
            uint32_t c0[LOADERS], c1[LOADERS];
            uint32_t n = 0;
#pragma unroll
            for (int l = 0; l < LOADERS; ++l) {
                c0[l] = phases(v0[l], s);
                c1[l] = phases(v1[l], s);
                n = max(n, max(c0[l], c1[l]));
            }
            if (n == 0) continue;
#pragma unroll
            for (int l = 0; l < LOADERS; ++l) {
                const uint32_t txl = loader_bytes<C>(l);
                if (c0[l] < n) {
                    if (PAIRED && c1[l] == n)
                        mbar_arrive_expect_tx(&full_bar[s], txl);
                    else
                        mbar_arrive(&full_bar[s]);
                } else if (PAIRED && c1[l] < n) {
                    mbar_complete_tx(&full_bar[s], txl);
                }
            }
            mbar_drain(&full_bar[s], (n - 1) & 1u);
        }
    }
    __syncthreads();
    // neither CTA of a pair leaves while the other may still target it
    if (PAIRED) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<C::PAIR>(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    // looked up once (thread-safe static initialisation)
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return nullptr;
    }();
    return fn;
}

// uint8 tensor map with 128-byte swizzled boxes of box_rows x 128 bytes.
bool make_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
              const cuuint64_t *strides, cuuint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint32_t box[3] = {128, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void *>(base),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// uint8 tensor map over `bytes` bytes viewed as rows of 256 bytes (no
// swizzle), boxes of box_rows rows: the scale buffers, whose 512-byte atoms
// are two such rows.
bool make_flat_map(CUtensorMap *m, const void *base, int64_t bytes, cuuint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int64_t rows = bytes / 256 > 0 ? bytes / 256 : 1;
    cuuint64_t dims[2] = {256, (cuuint64_t)rows};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// uint8 tensor map over the B scales viewed as [row blocks][2 kv_atoms rows
// of 256 bytes] (no swizzle): boxes of box_rows rows of box_rb consecutive
// row blocks, so one copy brings a stage's scale atoms of every B row block
// of a tile.
bool make_sfb_map(CUtensorMap *m, const void *base, int64_t row_blocks, int64_t kv_atoms,
                  cuuint32_t box_rows, cuuint32_t box_rb) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {256, (cuuint64_t)(2 * kv_atoms), (cuuint64_t)row_blocks};
    cuuint64_t strides[2] = {256, (cuuint64_t)(kv_atoms * 512)};
    cuuint32_t box[3] = {256, box_rows, box_rb};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
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

template <int KIND, int EPI, int BN, int STAGES, int ACC_BUFS, int EPI_WARPS, int SF_WARPS = 1,
          int PAIR = 1, int SILU_TAB = 0>
cudaError_t run_gemm(const GemmArgs &a, cudaStream_t s) {
    using C = Cfg<KIND, EPI, BN, STAGES, ACC_BUFS, EPI_WARPS, SF_WARPS, PAIR, MOEQ_SF_LOADER,
                  SILU_TAB>;
    // the kernel's tile prefix holds at most C::MAXG groups
    if (a.groups.num_groups > C::MAXG) return cudaErrorInvalidValue;
    const int64_t kbytes = (KIND == kNvfp4 || KIND == kMxfp4) ? a.K / 2 : a.K;
    const int64_t T = a.groups.total_rows;
    const int64_t E = a.groups.num_experts;
    CUtensorMap tA, tB, tSFA, tSFB, tC;
    memset(&tSFA, 0, sizeof(tSFA));
    memset(&tSFB, 0, sizeof(tSFB));
    memset(&tC, 0, sizeof(tC));
    cuuint64_t da[2] = {(cuuint64_t)kbytes, (cuuint64_t)T};
    cuuint64_t sa[1] = {(cuuint64_t)kbytes};
    cuuint64_t db[3] = {(cuuint64_t)kbytes, (cuuint64_t)a.N, (cuuint64_t)E};
    cuuint64_t sb[2] = {(cuuint64_t)kbytes, (cuuint64_t)(kbytes * a.N)};
    if (!make_map(&tA, a.a, 2, da, sa, C::BM)) return cudaErrorInvalidValue;
    if (!make_map(&tB, a.b, 3, db, sb, C::B_ROWS_CTA)) return cudaErrorInvalidValue;
    if (PAIR > 1 && C::SCALED) {
        const int64_t kv_atoms = a.K / C::SF_VEC / 4;
        const int64_t sfa_bytes = a.groups.scale_rows_total / 128 * kv_atoms * 512;
        const int64_t sfb_bytes = E * ((a.N + 127) / 128) * kv_atoms * 512;
        if (!make_flat_map(&tSFA, a.a_sf, sfa_bytes, 2 * C::SF_ATOMS)) return cudaErrorInvalidValue;
        if (!make_sfb_map(&tSFB, a.b_sf, E * ((a.N + 127) / 128), kv_atoms, 2 * C::SF_ATOMS, C::RB))
            return cudaErrorInvalidValue;
        (void)sfb_bytes;
    }
    if (C::EPI_BUF_BYTES) {
        // bf16 output [T, N], boxes of 32 rows x 32 columns (64 bytes) in
        // the staging buffer's 64-byte swizzle
        EncodeTiledFn enc = encode_fn();
        if (!enc) return cudaErrorInvalidValue;
        cuuint64_t dc[2] = {(cuuint64_t)a.N, (cuuint64_t)T};
        cuuint64_t sc[1] = {(cuuint64_t)a.N * 2};
        cuuint32_t bc[2] = {32, 32};
        cuuint32_t ec[2] = {1, 1};
        if (enc(&tC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.c, dc, sc, bc, ec,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    Params p;
    p.a_offsets = a.groups.row_offsets;
    p.a_sf_offsets = a.groups.scales_offsets;
    p.expert_ids = a.groups.expert_ids;
    p.num_groups = a.groups.num_groups;
    p.num_experts = a.groups.num_experts;
    p.total_rows = T;
    p.scale_rows_total = a.groups.scale_rows_total;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.a_scales = a.a_scales;
    p.b_scales = a.b_scales;
    p.a_sf = a.a_sf;
    p.b_sf = a.b_sf;
    p.expert_scales = a.expert_scales;
    p.out_tensor_scale = a.out_tensor_scale;
    p.row_scales = a.row_scales;
    p.c = reinterpret_cast<uint16_t *>(a.c);
    p.c_packed = a.c_packed;
    p.c_sf = a.c_sf;
    p.err = a.err;
    const int64_t nb = (a.N + BN - 1) / BN;
    // upper bound of the tiles (pair tiles for PAIR > 1) the offsets can give
    const int64_t tiles_ub = (T / (C::BM * PAIR) + a.groups.num_groups) * nb;
    auto kern = grouped_gemm_kernel<C, KIND, EPI>;
    // per-device launch set-up of this kernel, done once (the shared-memory
    // attribute and, for pairs, the resident cluster count)
    static std::atomic<int> attr_done[kMaxDevices];
    static std::atomic<int> max_cl_cache[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaError_t attr_err = cudaSuccess;
    cached_per_device(attr_done, dev, [&]() {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
        if (attr_err == cudaSuccess && C::NREG) {
            // the register split assumes the block holds THREADS x
            // LAUNCH_REGS registers: refuse to launch a build that differs
            cudaFuncAttributes fa;
            attr_err = cudaFuncGetAttributes(&fa, kern);
            if (attr_err == cudaSuccess && fa.numRegs != C::LAUNCH_REGS)
                attr_err = cudaErrorInvalidConfiguration;
        }
        return attr_err == cudaSuccess ? 1 : 0;
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (PAIR == 1) {
        const int grid = (int)(tiles_ub < sm_count() ? (tiles_ub > 0 ? tiles_ub : 1) : sm_count());
        return launch_pdl(kern, grid, C::THREADS, C::SMEM_BYTES, s, tA, tB, tSFA, tSFB, tC, p);
    }
    // persistent CTA pairs (clusters of two): as many as can be resident
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = kPdl;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(sm_count() / PAIR * PAIR), 1, 1);
    cudaError_t occ_err = cudaSuccess;
    const int max_clusters = cached_per_device(max_cl_cache, dev, [&]() {
        int n = 0;
        occ_err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        return occ_err == cudaSuccess && n >= 1 ? n : 0;
    });
    if (occ_err != cudaSuccess) return occ_err;
    if (max_clusters < 1) return cudaErrorNotSupported;
    int64_t clusters = tiles_ub < max_clusters ? (tiles_ub > 0 ? tiles_ub : 1) : max_clusters;
    cfg.gridDim = dim3((unsigned)(clusters * PAIR), 1, 1);
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, tA, tB, tSFA, tSFB, tC, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

// Tile configurations (compile-time).  NVFP4: 128x256 tiles with one TMEM
// accumulator (256 columns) plus per-stage scale slots; the epilogue drains
// its columns to registers and frees TMEM before computing, so the next
// tile's MMAs start at once.  FP8: 128x256 tiles, two accumulators.
#ifndef MOEQ_FP8_BN
#define MOEQ_FP8_BN 256
#endif
#ifndef MOEQ_FP8_STAGES
#define MOEQ_FP8_STAGES 4
#endif
#ifndef MOEQ_FP8_EPI_WARPS
#define MOEQ_FP8_EPI_WARPS 4
#endif
#ifndef MOEQ_FP4_BN
#define MOEQ_FP4_BN 256
#endif
#ifndef MOEQ_FP4_STAGES
#define MOEQ_FP4_STAGES 4
#endif
#ifndef MOEQ_FP4_ACC_BUFS
#define MOEQ_FP4_ACC_BUFS 1
#endif
#ifndef MOEQ_FP4_EPI_WARPS
#define MOEQ_FP4_EPI_WARPS 8
#endif
// Epilogue warps of the fused SwiGLU kernels: 8 (two per SM sub-partition,
// 128 accumulator columns each) leave more issue slots to the MMA and
// scale-copy warps than 16 (fused NVFP4 0.716 vs 0.757 ms on the 128-expert
// workload, with the SiLU in fused multiply-adds).
#ifndef MOEQ_SWIGLU_EPI_WARPS
#define MOEQ_SWIGLU_EPI_WARPS 8
#endif
// Warps issuing the shared -> TMEM scale copies (atoms dealt round-robin).
// Two, with the scale loads in the producer warp, is measured fastest on the
// 128-expert NVFP4 workload (fused 0.86 ms vs 1.00 ms with one copy warp and
// a scale-load warp; 3, 4 or 6 copy warps 1.07-1.09 ms, in earlier builds).
#ifndef MOEQ_SF_WARPS
#define MOEQ_SF_WARPS 2
#endif
// The fused NVFP4 kernel with the SiLU table (12 scale atoms per stage):
// six copy warps, 0.644-0.649 against 0.659-0.660 ms with two on the
// 128-expert workload; the MXFP4 one (6 atoms per stage) keeps two (0.634
// against 0.608 ms with six).
#ifndef MOEQ_SF_WARPS_NVFP4_TAB
#define MOEQ_SF_WARPS_NVFP4_TAB 6
#endif
// CTA-pair tiles (M = 256 over two SMs, tcgen05 cta_group::2, each SM
// staging half of the B tile) for the FP4 kinds: 0.78 vs 0.81 ms fused and
// 0.68 vs 0.74 ms bf16 out on the 128-expert NVFP4 workload.  Single-CTA
// tiles for FP8 rowwise (pairs: 1.294 vs 1.300 ms at MoE scale, 1.065 vs
// 0.964 ms on the decode shape).  MOEQ_GEMM_PAIR, when given, sets both.
#ifdef MOEQ_GEMM_PAIR
#define MOEQ_FP4_PAIR MOEQ_GEMM_PAIR
#define MOEQ_FP8_PAIR MOEQ_GEMM_PAIR
#endif
#ifndef MOEQ_FP4_PAIR
#define MOEQ_FP4_PAIR 2
#endif
#ifndef MOEQ_FP8_PAIR
#define MOEQ_FP8_PAIR 1
#endif
#ifndef MOEQ_FP4_PAIR_STAGES
#define MOEQ_FP4_PAIR_STAGES 5
#endif
#ifndef MOEQ_FP8_PAIR_STAGES
#define MOEQ_FP8_PAIR_STAGES 6
#endif
#ifndef MOEQ_MX8_STAGES
#define MOEQ_MX8_STAGES 6
#endif
// Fused SwiGLU epilogues of the FP4 kinds take silu(gate) from a
// shared-memory table (1) or compute it (0).
#ifndef MOEQ_SILU_TAB
#define MOEQ_SILU_TAB 1
#endif

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s) {
    constexpr int P = MOEQ_FP4_PAIR;
    constexpr int P8 = MOEQ_FP8_PAIR;
    constexpr int FP4_ST = P == 2 ? MOEQ_FP4_PAIR_STAGES : MOEQ_FP4_STAGES;
    constexpr int FP8_ST = P8 == 2 ? MOEQ_FP8_PAIR_STAGES : MOEQ_FP8_STAGES;
    if (a.kind == kFp8Rowwise && a.epi == kBf16) {
        if (a.N >= 256)
            return run_gemm<kFp8Rowwise, kBf16, MOEQ_FP8_BN, FP8_ST, 2, MOEQ_FP8_EPI_WARPS, 1, P8>(
                a, s);
        return run_gemm<kFp8Rowwise, kBf16, 64, 8, 2, 4>(a, s);
    }
    if (a.kind == kNvfp4 && a.epi == kBf16)
        return run_gemm<kNvfp4, kBf16, MOEQ_FP4_BN, FP4_ST, MOEQ_FP4_ACC_BUFS, MOEQ_FP4_EPI_WARPS,
                        MOEQ_SF_WARPS, P>(a, s);
    // fused SwiGLU on FP4: silu by table up to kSiluMaxGroups groups, computed
    // beyond (the same bytes either way)
    const bool tab = a.groups.num_groups <= kSiluMaxGroups;
    if (a.kind == kNvfp4 && a.epi == kSwiglu)
        return tab ? run_gemm<kNvfp4, kSwiglu, MOEQ_FP4_BN, FP4_ST, MOEQ_FP4_ACC_BUFS,
                              MOEQ_SWIGLU_EPI_WARPS,
                              MOEQ_SILU_TAB && P == 2 ? MOEQ_SF_WARPS_NVFP4_TAB : MOEQ_SF_WARPS, P,
                              MOEQ_SILU_TAB>(a, s)
                   : run_gemm<kNvfp4, kSwiglu, MOEQ_FP4_BN, FP4_ST, MOEQ_FP4_ACC_BUFS,
                              MOEQ_SWIGLU_EPI_WARPS, MOEQ_SF_WARPS, P>(a, s);
    if (a.kind == kMxfp4 && a.epi == kSwigluMx)
        return tab ? run_gemm<kMxfp4, kSwigluMx, MOEQ_FP4_BN, FP4_ST, MOEQ_FP4_ACC_BUFS,
                              MOEQ_SWIGLU_EPI_WARPS, MOEQ_SF_WARPS, P, MOEQ_SILU_TAB>(a, s)
                   : run_gemm<kMxfp4, kSwigluMx, MOEQ_FP4_BN, FP4_ST, MOEQ_FP4_ACC_BUFS,
                              MOEQ_SWIGLU_EPI_WARPS, MOEQ_SF_WARPS, P>(a, s);
    if (a.kind == kMxfp8 && a.epi == kSwigluMx)
        return run_gemm<kMxfp8, kSwigluMx, 128, MOEQ_MX8_STAGES, 2, 8>(a, s);
    if (a.kind == kMxfp4 && a.epi == kBf16)
        return run_gemm<kMxfp4, kBf16, MOEQ_FP4_BN, FP4_ST, MOEQ_FP4_ACC_BUFS, MOEQ_FP4_EPI_WARPS,
                        MOEQ_SF_WARPS, P>(a, s);
    if (a.kind == kMxfp8 && a.epi == kBf16)
        return run_gemm<kMxfp8, kBf16, 128, MOEQ_MX8_STAGES, 2, 4>(a, s);
    return cudaErrorNotSupported;
}

}  // namespace moeq
