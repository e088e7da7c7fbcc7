// Device-side building blocks shared by the moeq kernels (sm_103a):
// element codecs, the deterministic exp/SiLU, mbarrier / TMA / tcgen05
// wrappers written as inline PTX, and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moeq.h"

namespace moeq {

// ------------------------------------------------------------------ errors

__device__ __forceinline__ void set_error(uint32_t *err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

// Store guard.  Debug builds (MOEQ_DEBUG_BOUNDS) check every global store of
// the kernels against its buffer's extent first: a store outside it is
// skipped and sets MOEQ_DEVERR_BOUNDS.  Release builds compile the check out.
__device__ __forceinline__ bool store_ok(bool in_bounds, uint32_t *err) {
#ifdef MOEQ_DEBUG_BOUNDS
    if (!in_bounds) set_error(err, MOEQ_DEVERR_BOUNDS);
    return in_bounds;
#else
    (void)in_bounds;
    (void)err;
    return true;
#endif
}

// ------------------------------------------------- programmatic launches

// Every kernel of the library is launched with programmatic stream
// serialisation (launch_pdl below): its CTAs may be scheduled while the
// kernel before it in the stream is still finishing.  Each kernel therefore
// executes pdl_wait() in every thread before its first global memory access
// (read or write) -- the wait returns once the preceding grid has completed
// and its memory operations are visible, so the stream order of all memory
// effects is unchanged -- and pdl_trigger() once its own CTA no longer needs
// the SM to itself, which lets the next kernel's CTAs launch as this
// kernel's CTAs drain.  In a kernel launched without the attribute both are
// no-ops.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Compile-time switch: MOEQ_NO_PDL launches every kernel in plain stream
// order (the waits and triggers then do nothing).
#ifdef MOEQ_NO_PDL
constexpr int kPdl = 0;
#else
constexpr int kPdl = 1;
#endif

// Launches kern<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialisation; returns the launch status.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = kPdl;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ------------------------------------------------------------------ codecs

// bf16 bits -> fp32 (exact).
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) {
    return __uint_as_float(b << 16);
}

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return (uint32_t)__bfloat16_as_ushort(h);
}

// Eight fp32 -> eight E2M1 codes packed in 32 bits, element i in nibble i
// (round to nearest even, saturating).  cvt.*x2 puts its first source in the
// high half of the result, so each pair is given (x[2i+1], x[2i]).
__device__ __forceinline__ uint32_t e2m1x8(const float (&x)[8]) {
    uint32_t r;
    asm("{\n\t"
        ".reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t"
        "}"
        : "=r"(r)
        : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]),
          "f"(x[6]), "f"(x[7]));
    return r;
}

// Two fp32 -> two E4M3 codes in 16 bits, lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

__device__ __forceinline__ uint32_t e4m3(float x) { return e4m3x2(x, 0.0f) & 0xFFu; }

// Value of a non-negative finite E4M3 code (exact).
__device__ __forceinline__ float e4m3_pos_value(uint32_t code) {
    uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
    if (e == 0) return (float)m * 0.001953125f;            // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// ------------------------------------------- paired fp32 arithmetic (f32x2)
// Two independent IEEE fp32 operations per instruction (round to nearest
// even, subnormals kept): each lane gives exactly the scalar result.
struct F2 {
    uint64_t v;
};

__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float f2_lo(F2 a) {
    float lo;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {%0, t}, %1;\n\t}" : "=f"(lo) : "l"(a.v));
    return lo;
}

__device__ __forceinline__ float f2_hi(F2 a) {
    float hi;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {t, %0}, %1;\n\t}" : "=f"(hi) : "l"(a.v));
    return hi;
}

__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
    F2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}

__device__ __forceinline__ F2 add2(F2 a, F2 b) {
    F2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}

__device__ __forceinline__ F2 sub2(F2 a, F2 b) {
    F2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}

// Two fp32 -> bf16 (round to nearest even) -> fp32.
__device__ __forceinline__ F2 round_bf16_2(F2 a) {
    uint32_t b;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(f2_hi(a)), "f"(f2_lo(a)));
    return f2(__uint_as_float(b << 16), __uint_as_float(b & 0xFFFF0000u));
}

// ------------------------------------------------------- NVFP4 block rule
// One 16-element block: amax m, per-expert inverse tensor scale inv.
// sb = E4M3((m * inv) / 6); r = inv / sb; codes = E2M1(x * r) (all +0 when
// sb == 0).  Every step is one IEEE fp32 operation (no contraction).
struct Nvfp4Scale {
    uint32_t code;  // E4M3 scale code
    float r;        // element multiplier, 0 when the block scale is 0
};

__device__ __forceinline__ Nvfp4Scale nvfp4_block_scale(float m, float inv) {
    float sbf = __fdiv_rn(__fmul_rn(m, inv), 6.0f);
    Nvfp4Scale s;
    s.code = e4m3(sbf);
    float sb = e4m3_pos_value(s.code);
    s.r = (sb == 0.0f) ? 0.0f : __fdiv_rn(inv, sb);
    return s;
}

// The E4M3 scale code of a block only (the element multiplier is then
// inv / value(code), which callers may tabulate per code).
__device__ __forceinline__ Nvfp4Scale nvfp4_block_scale_code(float m, float inv) {
    Nvfp4Scale s;
    s.code = e4m3(__fdiv_rn(__fmul_rn(m, inv), 6.0f));
    s.r = 0.0f;
    return s;
}


// Eight elements of a block -> 32 bits of packed codes (the products x * r
// in paired multiplies: the same IEEE products as scalar code).
__device__ __forceinline__ uint32_t nvfp4_codes8(const float (&x)[8], float r) {
    if (r == 0.0f) return 0u;
    const F2 r2 = f2(r, r);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const F2 q = mul2(f2(x[i], x[i + 1]), r2);
        y[i] = f2_lo(q);
        y[i + 1] = f2_hi(q);
    }
    return e2m1x8(y);
}

// ------------------------------------------------------- MX block rule
// Scale code of an MX block whose amax m is a positive fp32 value: the OCP
// floor rule c = clamp(floor(log2 m) - emax + 127, 0, 254), floor(log2 m)
// read from the fp32 exponent bits (subnormals included).  For finite m,
// c <= 252 (emax >= 2), so the element multiplier 2^(127 - c) is a normal
// fp32 number.
__device__ __forceinline__ uint32_t mx_scale_code_f32(float m, int emax) {
    const uint32_t b = __float_as_uint(m);
    const int ef = (int)((b >> 23) & 0xFFu);
    const int e = ef > 0 ? ef - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
    return (uint32_t)min(max(e - emax + 127, 0), 254);
}

__device__ __forceinline__ float mx_multiplier(uint32_t c) {
    return __uint_as_float((254u - c) << 23);  // 2^(127 - c)
}

// ------------------------------------------------ deterministic exp / SiLU
// The library's SiLU, silu(g) = g * sigma(g), is defined by the steps below,
// each one IEEE fp32 operation or one fused multiply-add (a single
// rounding), so that every kernel reproduces it bit for bit:
//   e     = exp(-|g|): Cody-Waite reduction x = n ln2 + f with ln 2 split
//           into a 16-significant-bit head (45426 / 2^16) and an fp32 tail,
//           the degree-7 Taylor polynomial of e^f by Horner's rule, then
//           p * 2^n with 2^n taken as 0 for n < -126 (x clamped to >= -104);
//   d     = 1 + e, in [1, 2];
//   r     = 1 / d: Newton-Raphson from the minimax line 24/17 - 8/17 d,
//           three steps q = 1 - d r, r = r + r q;
//   sigma = r for g >= 0, e * r otherwise (e / (1 + e) = 1 / (1 + e^-g)).
// All of it runs two values at a time in paired arithmetic.

__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
    F2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return d;
}

__device__ __forceinline__ F2 f2s(float x) { return f2(x, x); }

// e^x of two arguments x <= 0 (a NaN argument gives 0).
__device__ __forceinline__ F2 exp_neg2(float x0, float x1) {
    const float kLog2e = 1.44269502162933349609375f;      // fp32(1 / ln 2)
    const float kLn2Hi = 0.693145751953125f;              // 45426 / 65536
    const float kLn2Lo = 1.428606765330187045037746429443359375e-06f;
    const float kShift = 12582912.0f;                     // 1.5 * 2^23
    const float c[8] = {1.0f, 1.0f, 0.5f,
                        0.16666667163372039794921875f,          // fp32(1/3!)
                        0.0416666679084300994873046875f,        // fp32(1/4!)
                        0.008333333767950534820556640625f,      // fp32(1/5!)
                        0.001388888922519981861114501953125f,   // fp32(1/6!)
                        0.0001984127011382952332496643066406f}; // fp32(1/7!)
    const F2 xc = f2(fmaxf(x0, -104.0f), fmaxf(x1, -104.0f));
    // t = 1.5 * 2^23 + n, n = x log2(e) rounded to an integer (ties to even)
    const F2 t = fma2(xc, f2s(kLog2e), f2s(kShift));
    const F2 n = sub2(t, f2s(kShift));
    F2 f = fma2(n, f2s(-kLn2Hi), xc);
    f = fma2(n, f2s(-kLn2Lo), f);
    F2 p = f2s(c[7]);
#pragma unroll
    for (int k = 6; k >= 0; --k) p = fma2(p, f, f2s(c[k]));
    // the bits of t are 0x4B400000 + n (n in [-150, 0]): shifted left by 23
    // they give the exponent field n (mod 2^32); the fp32 bits of 2^n are
    // (n + 127) << 23, negative (then clamped to +0) for n < -126
    const int s0 = max((int)((__float_as_uint(f2_lo(t)) << 23) + (127u << 23)), 0);
    const int s1 = max((int)((__float_as_uint(f2_hi(t)) << 23) + (127u << 23)), 0);
    return mul2(p, f2(__int_as_float(s0), __int_as_float(s1)));
}

// silu(g) = g * sigma(g) for two gates.
__device__ __forceinline__ F2 silu2(float g0, float g1) {
    const float kSeedA = 1.41176474094390869140625f;      // fp32(24 / 17)
    const float kSeedB = 0.4705882370471954345703125f;    // fp32(8 / 17)
    const F2 e = exp_neg2(-fabsf(g0), -fabsf(g1));
    const F2 nd = sub2(f2s(-1.0f), e);                    // -d = -(1 + e)
    F2 r = fma2(nd, f2s(kSeedB), f2s(kSeedA));
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const F2 q = fma2(nd, r, f2s(1.0f));
        r = fma2(r, q, r);
    }
    const F2 er = mul2(e, r);
    const F2 sg = f2(g0 >= 0.0f ? f2_lo(r) : f2_lo(er), g1 >= 0.0f ? f2_hi(r) : f2_hi(er));
    return mul2(f2(g0, g1), sg);
}

// h = silu(g) * u for two (gate, up) pairs.
__device__ __forceinline__ F2 swiglu2(float g0, float g1, float u0, float u1) {
    return mul2(silu2(g0, g1), f2(u0, u1));
}

// SiLU of bf16 gates by table.  The table holds silu(g), computed by silu2,
// for every bf16 g whose biased exponent lies in [kSiluE0, kSiluE0 +
// kSiluExps), positive gates first, then their negative twins (2 x 4096
// fp32).  Outside that range the definition reduces exactly (checked for
// every bf16 value) to silu(g) = g * 1/2 below it (sigma = 1/2 to fp32
// precision, zero and subnormals included) and to g * (g >= 0 ? 1 : 0)
// above it (sigma = 1 or 0; inf and NaN as the definition gives them).
constexpr uint32_t kSiluE0 = 102, kSiluExps = 32;
constexpr uint32_t kSiluHalf = kSiluExps * 128;           // entries per sign
constexpr uint32_t kSiluTableBytes = 2 * kSiluHalf * 4;

// Fills the table; every thread of the CTA calls it (a CTA barrier must
// follow before the table is read).
__device__ __forceinline__ void build_silu_table(float *tab) {
    for (uint32_t i = threadIdx.x; i < kSiluHalf; i += blockDim.x) {
        const uint32_t gb = (kSiluE0 << 7) + i;
        const F2 sv = silu2(__uint_as_float(gb << 16), __uint_as_float((gb | 0x8000u) << 16));
        tab[i] = f2_lo(sv);
        tab[kSiluHalf + i] = f2_hi(sv);
    }
}

// silu(g) for the bf16 gate with bits gb (low 16 bits).
__device__ __forceinline__ float silu_lookup(uint32_t gb, const float *tab) {
    const uint32_t mag = gb & 0x7FFFu;
    const uint32_t t = mag - (kSiluE0 << 7);
    const float g = __uint_as_float(gb << 16);
    if (t < kSiluHalf) return tab[t + ((gb & 0x8000u) ? kSiluHalf : 0u)];
    return mag < (kSiluE0 << 7) ? __fmul_rn(g, 0.5f) : __fmul_rn(g, g >= 0.0f ? 1.0f : 0.0f);
}

// silu_lookup with the table at shared-memory address tab, read by an
// explicit shared load (issued only for gates inside the band): the same
// entries and closed forms.
__device__ __forceinline__ float silu_lookup_shared(uint32_t gb, uint32_t tab) {
    const uint32_t mag = gb & 0x7FFFu;
    const uint32_t t = mag - (kSiluE0 << 7);
    const float g = __uint_as_float(gb << 16);
    if (t < kSiluHalf) {
        float v;
        asm volatile("ld.shared.f32 %0, [%1];"
                     : "=f"(v)
                     : "r"(tab + 4u * (t + ((gb & 0x8000u) ? kSiluHalf : 0u))));
        return v;
    }
    return mag < (kSiluE0 << 7) ? __fmul_rn(g, 0.5f) : __fmul_rn(g, g >= 0.0f ? 1.0f : 0.0f);
}

// h = silu(g) * u for two (gate, up) words (gate bits in the low half, up
// in the high half), silu by table.
__device__ __forceinline__ F2 swiglu2_tab(uint32_t w0, uint32_t w1, const float *tab) {
    return mul2(f2(silu_lookup(w0 & 0xFFFFu, tab), silu_lookup(w1 & 0xFFFFu, tab)),
                f2(__uint_as_float(w0 & 0xFFFF0000u), __uint_as_float(w1 & 0xFFFF0000u)));
}

// ----------------------------------------------------- tiled scale layout
// Byte offset of the 4-byte word holding scale columns [4 kb, 4 kb + 4) of
// logical row r, for kv_atoms = ceil(Kv / 4) atom columns.
__device__ __forceinline__ int64_t sf_word_offset(int64_t r, int64_t kb, int64_t kv_atoms) {
    return ((r >> 7) * kv_atoms + kb) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

// ------------------------------------------------------------ group search
// Largest g in [0, G) with offs[g] <= x (offs non-decreasing, offs[0] <= x).
__device__ __forceinline__ int upper_bound_minus1(const uint32_t *offs, int G, uint32_t x) {
    int lo = 0, hi = G;  // invariant: offs[lo] <= x, answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(offs + mid) <= x) lo = mid; else hi = mid;
    }
    return lo;
}

// ------------------------------------------------------------ PTX: memory

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Completes `bytes` of the transaction count of the barrier's current
// phase without a copy (for copies that were announced but never issued).
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// CLUSTER: acquire at cluster scope, for barriers that the other CTA of a
// pair arrives on (its copies, commits or remote arrivals).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    return ok != 0;
}

// ~1 s at the GB300's maximum SM clock.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when *abort is set by another role, or after
// kWaitLimitCycles, in which case it sets the timeout bit and *abort.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          uint32_t *err) {
    uint32_t a = smem_u32(bar);
    if (mbar_try_wait<CLUSTER>(a, parity)) return true;
    long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait<CLUSTER>(a, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            set_error(err, MOEQ_DEVERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Waits for a phase with a bound but without consulting the abort flag;
// used only to drain in-flight asynchronous work before the CTA exits.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    uint32_t a = smem_u32(bar);
    long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) break;
    }
}

// TMA tiled loads into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// CTA-pair variants (.cta_group::2): the box lands in this CTA's shared
// memory and completes on a barrier given by its shared::cluster address,
// which may be the barrier of the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar,
                                                 int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t bar,
                                                 int x, int y, int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// shared::cluster address of the variable at shared::cta address `a` in
// the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// 32-bit load from the shared memory of a CTA of the cluster (address from
// mapa_shared).
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Arrival on a barrier given by its shared::cluster address (possibly in
// the other CTA of the pair), releasing at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

// Arrival without memory ordering, for an accumulator release: the arriving
// warp's tensor-memory loads have completed (tcgen05.wait::ld) before it
// arrives, and the waiter needs nothing else from it.  A release at cluster
// scope would first wait for every global store the warp has in flight.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Cluster-wide barrier: every thread of every CTA of the cluster arrives.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// --------------------------------------------------------- PTX: tcgen05

// CG = 1: this CTA's tensor memory; CG = 2: one warp of each CTA of a pair
// allocates collectively and both get the same address.  Every tcgen05
// operation of a kernel uses the same CG.
template <int CG = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    if (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(dst_smem)),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(dst_smem)),
                     "r"(ncols)
                     : "memory");
}

template <int CG = 1>
__device__ __forceinline__ void tmem_relinquish() {
    if (CG == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives on `bar` once every tcgen05 operation issued so far by this
// thread has completed.
template <int CG = 1>
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    if (CG == 1)
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_u32(bar))
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_u32(bar))
            : "memory");
}

// As tc_commit, arriving on the barrier at the same offset in every CTA of
// the cluster named in cta_mask.
template <int CG = 1>
__device__ __forceinline__ void tc_commit_mc(uint64_t *bar, uint16_t cta_mask) {
    if (CG == 1)
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::"
            "cluster.b64 [%0], %1;" ::"r"(smem_u32(bar)),
            "h"(cta_mask)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::"
            "cluster.b64 [%0], %1;" ::"r"(smem_u32(bar)),
            "h"(cta_mask)
            : "memory");
}

// Shared-memory matrix descriptor, K-major operand staged by TMA with 128B
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;              // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Descriptor of one 512-byte scale atom in shared memory for tcgen05.cp
// 32x128b: 32 rows of 16 bytes, no swizzle, 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptors (dense, K-major A and B, fp32 accumulator).
// kind::f8f6f4 with E4M3 x E4M3.
__host__ __device__ constexpr uint32_t idesc_f8_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// kind::mxf4nvf4, E2M1 x E2M1 with UE4M3 scales (16-element blocks).
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// kind::mxf8f6f4, E4M3 x E4M3 with UE8M0 scales; sf_id picks the byte of
// the 32-bit scale cell (the 32-element block within four).
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int M, int N, int sf_id) {
    return ((uint32_t)sf_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_id << 29);
}

// kind::mxf4, E2M1 x E2M1 with UE8M0 scales (32-element blocks); sf_id 0 or
// 2 picks the byte pair of the scale cell (two blocks per K=64 step).
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, int sf_id) {
    return ((uint32_t)sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           (1u << 23) | ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_id << 29);
}

template <int CG = 1>
__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, "
            "[%4], [%5], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, "
            "[%4], [%5], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}

// CG = 2: issued by one thread of the even CTA of a pair; A rows and the B
// rows of each half come from the shared memory of each CTA at the same
// offsets, and each CTA's tensor memory receives its half of the rows of D.
template <int CG = 1>
__device__ __forceinline__ void mma_f8f6f4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
            : "memory");
}

template <int CG = 1>
__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
            "[%4], [%5], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
            "[%4], [%5], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}

template <int CG = 1>
__device__ __forceinline__ void mma_mxf8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
            "[%4], [%5], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
            "[%4], [%5], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}

// Copies one 512-byte scale atom (32 rows x 16 bytes) from shared memory to
// 4 TMEM columns, replicated into all four 32-lane quarters.  CG = 2: each
// CTA of the pair copies the atom at this offset of its own shared memory.
template <int CG = 1>
__device__ __forceinline__ void tmem_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
    if (CG == 1)
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                     : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                     : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Streaming 16-byte load of read-once data (not kept in L1).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// --------------------------------------------------------- global stores

__device__ __forceinline__ void st_global_v4(void *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

}  // namespace moeq
