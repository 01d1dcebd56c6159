// kvd_common.cuh — device helpers shared by the kernels of the paged decode library.
//
// Inline PTX for sm_103a: mbarrier, 1-D bulk copy (TMA engine, no tensor map),
// warp-level tensor-core MMA (m16n8k16), movmatrix, ex2, %globaltimer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/kvd.h"

namespace kvd {

constexpr int kDh = 128;          // head dimension
constexpr int kBs = 16;           // tokens per block
constexpr int kMaxG = 8;          // query heads per KV head (one MMA n-tile)
constexpr int kMaxBatch = 2048;
constexpr int kTileBf16 = kBs * kDh * 2;   // 4096 bytes
constexpr int kTileFp8 = kBs * kDh;        // 2048 bytes
constexpr int kScaleBytes = 2 * kBs * 4;   // FP8 record tail: K and V scales per slot
constexpr int kRecordBf16 = 2 * kTileBf16;                 // 8192 bytes
constexpr int kRecordFp8 = 2 * kTileFp8 + kScaleBytes;     // 4224 bytes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;

// Storage format of one block's K/V: BF16 values, or 8-bit codes (E4M3 / E5M2) with one fp32
// scale per (token, KV head) for K and one for V.
constexpr int kFmtBf16 = 0, kFmtE4m3 = 1, kFmtE5m2 = 2;
// Internal format of a per-block precision byte of a mixed pool (KVD_BF16, KVD_FP8_E4M3 or
// KVD_FP8_E5M2), or -1 for any other value.
__host__ __device__ __forceinline__ int block_format(int code) {
    return code == KVD_BF16 ? kFmtBf16 : code == KVD_FP8_E4M3 ? kFmtE4m3 : code == KVD_FP8_E5M2 ? kFmtE5m2 : -1;
}

// ---------------------------------------------------------------- fragment order
// A 16-token × 128-dim tile is stored so that lane `lane` of a warp finds the
// A-operand fragment of k-step (or m-tile) i of mma.m16n8k16 in one 16-byte
// (BF16) or 8-byte (FP8) chunk.  K feeds S^T = K·Q^T (rows = tokens,
// cols = dims); V feeds O^T = V^T·P^T (rows = dims, cols = tokens).
__host__ __device__ __forceinline__ int k_frag_i(int t, int d, int* lane, int* e) {
    int c = d & 15;
    *lane = ((t & 7) << 2) | ((c & 7) >> 1);
    *e = (c & 1) | ((t >> 3) << 1) | ((c >> 3) << 2);
    return d >> 4;
}
__host__ __device__ __forceinline__ int v_frag_i(int t, int d, int* lane, int* e) {
    int r = d & 15;
    *lane = ((r & 7) << 2) | ((t & 7) >> 1);
    *e = (t & 1) | ((r >> 3) << 1) | ((t >> 3) << 2);
    return d >> 4;
}
__host__ __device__ __forceinline__ int bf16_tile_index(int i, int lane, int e) { return ((i * 32 + lane) << 3) | e; }
__host__ __device__ __forceinline__ int fp8_tile_index(int i, int lane, int e) {
    return ((((i >> 1) * 32 + lane) << 4) | ((i & 1) << 3) | e);
}

// ------------------------------------------------------------------ error word
__device__ __forceinline__ void report(int32_t* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// -------------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete, giving up after
// `limit_ns` nanoseconds or as soon as *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------- bulk copy (TMA)
// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.  Both
// addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// A logit written for the score update: kept in L2 (evict-last) until the score kernel, which runs
// about one layer later, reads it, so neither the write nor the read reaches DRAM.
__device__ __forceinline__ void st_logit(float* p, float v) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
        "st.global.L2::cache_hint.f32 [%0], %1, pol;\n\t}" ::"l"(p), "f"(v)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// --------------------------------------------------------------- tensor cores
__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Transpose an 8x8 matrix of 16-bit elements held one row per 4 lanes.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The two bf16 halves of a packed pair as floats (lo, hi).
__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&v);
    return __bfloat1622float2(h);
}

// The two f16 halves of a packed pair as floats (lo, hi).
__device__ __forceinline__ float2 unpack_f16(uint32_t v) {
    const __half2 h = *reinterpret_cast<const __half2*>(&v);
    return __half22float2(h);
}
// Two E4M3 codes (low byte = lower element) -> f16x2 in one instruction; exact, since
// every E4M3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
    uint32_t r;
    const uint16_t v = static_cast<uint16_t>(v16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// Write one token's K and V rows (128 bf16 each) into slot t of a pool record, by one
// warp: lane l holds dims 4l..4l+3.  BF16 records (FMT kFmtBf16) store the values in
// fragment order; 8-bit records store code(x / scale) with scale = fp32(absmax/top) (1 for a
// zero row), top = 448 (E4M3) or 57,344 (E5M2), the largest finite value of the format,
// codes rounded to nearest even and saturated, per K and per V, the scales after the two tiles.
// ANGLE (E4M3 only): the K row's word after the tiles is its logit factor instead of its scale,
// w = fp32(half(||k||) / ||d||) with d the values of its codes, in fp64 (0 for a zero row); the
// direction code is the codes themselves (they depend on k/||k|| only).
template <int FMT, bool ANGLE = false>
__device__ __forceinline__ void write_token(uint8_t* record, int t, const uint16_t* krow, const uint16_t* vrow,
                                            int lane) {
    constexpr bool FP8 = FMT != kFmtBf16;
    const uint2 kraw = *reinterpret_cast<const uint2*>(krow + lane * 4);
    const uint2 vraw = *reinterpret_cast<const uint2*>(vrow + lane * 4);
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kraw);
    const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vraw);
    if constexpr (!FP8) {
        __nv_bfloat16* ktile = reinterpret_cast<__nv_bfloat16*>(record);
        __nv_bfloat16* vtile = ktile + kBs * kDh;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = lane * 4 + j;
            int fl, fe;
            int i = k_frag_i(t, d, &fl, &fe);
            ktile[bf16_tile_index(i, fl, fe)] = kb[j];
            i = v_frag_i(t, d, &fl, &fe);
            vtile[bf16_tile_index(i, fl, fe)] = vb[j];
        }
    } else {
        float kx[4], vx[4];
        float kmax = 0.f, vmax = 0.f;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            kx[j] = __bfloat162float(kb[j]);
            vx[j] = __bfloat162float(vb[j]);
            kmax = fmaxf(kmax, fabsf(kx[j]));
            vmax = fmaxf(vmax, fabsf(vx[j]));
        }
        #pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kmax = fmaxf(kmax, __shfl_xor_sync(kFull, kmax, o));
            vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
        }
        constexpr float kTop = FMT == kFmtE5m2 ? 57344.f : 448.f;
        constexpr __nv_fp8_interpretation_t kInterp = FMT == kFmtE5m2 ? __NV_E5M2 : __NV_E4M3;
        const float ks = (kmax == 0.f) ? 1.f : __fdiv_rn(kmax, kTop);
        const float vs = (vmax == 0.f) ? 1.f : __fdiv_rn(vmax, kTop);
        uint8_t* ktile = record;
        uint8_t* vtile = record + kTileFp8;
        double r2 = 0.0, d2 = 0.0;   // ANGLE: squared radius and squared code norm, this lane's dims
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = lane * 4 + j;
            const uint8_t kc = __nv_cvt_float_to_fp8(__fdiv_rn(kx[j], ks), __NV_SATFINITE, kInterp);
            const uint8_t vc = __nv_cvt_float_to_fp8(__fdiv_rn(vx[j], vs), __NV_SATFINITE, kInterp);
            int fl, fe;
            int i = k_frag_i(t, d, &fl, &fe);
            ktile[fp8_tile_index(i, fl, fe)] = kc;
            i = v_frag_i(t, d, &fl, &fe);
            vtile[fp8_tile_index(i, fl, fe)] = vc;
            if constexpr (ANGLE) {
                const double c = static_cast<double>(__half2float(__half(__nv_cvt_fp8_to_halfraw(kc, __NV_E4M3))));
                r2 += static_cast<double>(kx[j]) * static_cast<double>(kx[j]);
                d2 += c * c;   // exact: code values are multiples of 2^-9 below 2^9
            }
        }
        float kw = ks;
        if constexpr (ANGLE) {
            #pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                r2 += __shfl_xor_sync(kFull, r2, o);
                d2 += __shfl_xor_sync(kFull, d2, o);
            }
            __half rh = __double2half(__dsqrt_rn(r2));
            if (__hisinf(rh)) rh = __ushort_as_half(0x7BFFu);
            kw = d2 > 0.0 ? __double2float_rn(__ddiv_rn(static_cast<double>(__half2float(rh)), __dsqrt_rn(d2))) : 0.f;
        }
        if (lane == 0) {
            float* sc = reinterpret_cast<float*>(record + 2 * kTileFp8);
            sc[t] = kw;
            sc[kBs + t] = vs;
        }
    }
}

// ------------------------------------------------------------------ low-bit records
// A low-bit record holds BITS-wide codes (4 or 2) of the K tile and of the V tile, then for K
// and for V a table [16 tokens][NG groups] of (scale, zero point) half-precision pairs (scale in
// the low 16 bits); a value reads back as code·scale + zero.  A group is 128/NG consecutive
// dims of one token's row.
__host__ __device__ constexpr int lowbit_tile_bytes(int bits) { return kBs * kDh * bits / 8; }
__host__ __device__ constexpr int lowbit_meta_bytes(int ng) { return kBs * ng * 4; }
__host__ __device__ constexpr int lowbit_record_bytes(int bits, int ng) {
    return 2 * lowbit_tile_bytes(bits) + 2 * lowbit_meta_bytes(ng);
}

// Code placement.  A byte holds 8/BITS codes of one token, in bit fields h·BITS (h < 8/BITS),
// for dims 16 apart: the same fragment position of 8/BITS consecutive k-steps (K) or m-tiles
// (V).  Masking field h of a word leaves one code in the low bits of each byte; as an E4M3
// byte such a code c < 16 decodes exactly to c·2^-9, so one cvt turns bytes (0,1) and one bytes
// (2,3) of the masked word into the f16 pairs of two fragment registers.  Words are grouped
// four to a 16-byte chunk, chunk-major then lane, so a warp reads a chunk conflict-free.
//   K (rows = tokens): word (kg, th) of lane = 4·(t%8) + tq holds token t = lane/4 + 8·th; byte
//     j, field h: dim 16·(P·kg + h) + 2·tq + (j%2) + 8·(j/2), P = 8/BITS.  Fragment registers
//     of k-step P·kg + h: a0 = bytes(0,1) of th 0, a1 = bytes(0,1) of th 1, a2/a3 = bytes(2,3).
//   V (rows = dims): word (kg, th) of lane = 4·r + tq holds tokens 2·tq + (j%2) + 8·th; byte j,
//     field h: dim 16·(P·kg + h) + r + 8·(j/2).  m-tile P·kg + h: a0 = bytes(0,1) of th 0,
//     a1 = bytes(2,3) of th 0, a2/a3 the same of th 1.
//   word index in the tile: ((kg/2)·32 + lane)·4 + (kg%2)·2 + th.
__host__ __device__ __forceinline__ int lowbit_word(int kg, int lane, int th) {
    return ((kg >> 1) * 32 + lane) * 4 + (kg & 1) * 2 + th;
}
// Byte of a K (V) tile that holds the code of token t, dim d; its field is (d/16) % (8/bits).
__host__ __device__ __forceinline__ int lowbit_k_byte(int bits, int t, int d) {
    const int kg = d / (16 * (8 / bits));
    const int c = d & 15;
    const int lane = 4 * (t & 7) + ((c & 7) >> 1);
    return lowbit_word(kg, lane, t >> 3) * 4 + ((c & 1) | ((c >> 3) << 1));
}
__host__ __device__ __forceinline__ int lowbit_v_byte(int bits, int t, int d) {
    const int kg = d / (16 * (8 / bits));
    const int r = d & 15;
    const int lane = 4 * (r & 7) + ((t & 7) >> 1);
    return lowbit_word(kg, lane, t >> 3) * 4 + ((t & 1) | ((r >> 3) << 1));
}

// Nearest half-precision value, saturated to ±65,504 instead of overflowing.
__device__ __forceinline__ __half half_sat(float v) {
    const __half h = __float2half_rn(v);
    if (__hisinf(h)) return __ushort_as_half(v > 0.f ? 0x7BFFu : 0xFBFFu);
    return h;
}

// Quantise one group of a row held LPG lanes × 4 values (a group = 4·LPG consecutive dims):
// mn, mx over the group; scale = half(fp32((mx − mn)/(2^BITS − 1))), 1 when that is 0;
// zero = half(mn); code = clamp(rint(fp32(fp32(x − zero)/scale)), 0, 2^BITS − 1), single
// precision, ties to even.  Returns the (scale, zero) bits packed as one word.
template <int BITS, int LPG>
__device__ __forceinline__ uint32_t lowbit_quantise(const float (&x)[4], int (&code)[4]) {
    constexpr float kTop = static_cast<float>((1 << BITS) - 1);
    float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    #pragma unroll
    for (int o = 1; o < LPG; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    }
    __half hs = half_sat(__fdiv_rn(__fsub_rn(mx, mn), kTop));
    if (__half2float(hs) == 0.f) hs = __float2half_rn(1.f);
    const __half hz = half_sat(mn);
    const float s = __half2float(hs), z = __half2float(hz);
    #pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float r = rintf(__fdiv_rn(__fsub_rn(x[k], z), s));
        code[k] = static_cast<int>(fminf(fmaxf(r, 0.f), kTop));
    }
    return static_cast<uint32_t>(__half_as_ushort(hs)) | (static_cast<uint32_t>(__half_as_ushort(hz)) << 16);
}

// Write one token's K and V rows into slot t of a low-bit record, by one warp (lane l holds
// dims 4l..4l+3).  A byte takes the codes of dims 16 apart from 8/BITS lanes; the lanes that
// own its first dim gather them by shuffles and store whole bytes, so tokens written at the
// same time never share a byte.
template <int BITS, int NG>
__device__ __forceinline__ void write_token_lowbit(uint8_t* record, int t, const uint16_t* krow, const uint16_t* vrow,
                                                   int lane) {
    constexpr int kLpg = 32 / NG;          // lanes per group
    constexpr int kPer = 8 / BITS;         // codes per byte
    constexpr int kTile = lowbit_tile_bytes(BITS);
    const uint2 kraw = *reinterpret_cast<const uint2*>(krow + lane * 4);
    const uint2 vraw = *reinterpret_cast<const uint2*>(vrow + lane * 4);
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kraw);
    const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vraw);
    float kx[4], vx[4];
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        kx[j] = __bfloat162float(kb[j]);
        vx[j] = __bfloat162float(vb[j]);
    }
    int kc[4], vc[4];
    const uint32_t ksz = lowbit_quantise<BITS, kLpg>(kx, kc);
    const uint32_t vsz = lowbit_quantise<BITS, kLpg>(vx, vc);
    uint32_t kp = 0, vp = 0;   // this lane's 4 codes, code j in bits BITS·j
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        kp |= static_cast<uint32_t>(kc[j]) << (BITS * j);
        vp |= static_cast<uint32_t>(vc[j]) << (BITS * j);
    }
    // field h of a byte comes from lane + 4h (dims 16h further on)
    uint32_t kf[kPer], vf[kPer];
    kf[0] = kp;
    vf[0] = vp;
    #pragma unroll
    for (int h = 1; h < kPer; ++h) {
        kf[h] = __shfl_down_sync(kFull, kp, 4 * h);
        vf[h] = __shfl_down_sync(kFull, vp, 4 * h);
    }
    if ((lane & (4 * kPer - 4)) == 0) {
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t kbyte = 0, vbyte = 0;
            #pragma unroll
            for (int h = 0; h < kPer; ++h) {
                kbyte |= ((kf[h] >> (BITS * j)) & ((1u << BITS) - 1)) << (BITS * h);
                vbyte |= ((vf[h] >> (BITS * j)) & ((1u << BITS) - 1)) << (BITS * h);
            }
            const int d = 4 * lane + j;
            record[lowbit_k_byte(BITS, t, d)] = static_cast<uint8_t>(kbyte);
            record[kTile + lowbit_v_byte(BITS, t, d)] = static_cast<uint8_t>(vbyte);
        }
    }
    if (lane % kLpg == 0) {
        const int gi = lane / kLpg;
        uint32_t* meta = reinterpret_cast<uint32_t*>(record + 2 * kTile);
        meta[t * NG + gi] = ksz;
        meta[kBs * NG + t * NG + gi] = vsz;
    }
}

// 16-byte asynchronous copy global → shared through the load path (any global address the
// GPU maps, host memory included).  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16_g2s(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Raise the mbarrier's pending count by one now and lower it once every cp.async this thread
// issued before has landed: the current phase cannot complete before those copies.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Order generic-proxy shared-memory writes before this thread's later bulk (async-proxy) copies.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Make this thread's generic-proxy global writes visible to its later bulk copies.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Programmatic dependent launch.  Every kernel of a decode call is launched as a
// programmatic dependent of the kernel before it in the stream and starts with pdl_wait(),
// which returns once that kernel has completed and its writes are visible (at once when
// there is no such kernel), so its CTAs can be resident before the predecessor ends.  The
// decode kernel signals its dependents once a CTA has streamed its last block; the small
// merge kernels signal at their start, so the next layer's decode CTAs are scheduled
// while the merge runs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Four E4M3 codes of one word -> two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi); the
// 16-bit halves are taken as register halves, so no shift or mask is issued.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// The same for four E5M2 codes (an E5M2 value is the upper byte of an f16 value).
__device__ __forceinline__ void e5m2x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, a;\n\t"
        "cvt.rn.f16x2.e5m2x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}
template <int FMT>
__device__ __forceinline__ void f8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if constexpr (FMT == kFmtE5m2) e5m2x4_to_f16x2x2(w, lo, hi);
    else e4m3x4_to_f16x2x2(w, lo, hi);
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace kvd
