// common.cuh -- device helpers shared by the quantizer and the convolution kernels.
//
//  * element-format traits and exact round-to-nearest of a real quotient
//    (MicroQonv §III-A: B_scale = CastE4M3(amax / (maxB_ef T_scale)),
//    X^q = Round(X / (B_scale T_scale))), built on the sm_100-family
//    conversion instructions plus an exact fma-sign tie-break;
//  * decode of one packed 8x8 block row into eight fp16 values (code x B_scale
//    is exact in fp16 for every format used here, see DecodeScale below);
//  * bounded mbarrier waits and the tcgen05 / TMEM PTX wrappers.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace mq {

// status bits, OR-ed into the device status word (mirror of mq_status values)
constexpr uint32_t ST_NONFINITE = 1u << 4;
constexpr uint32_t ST_TIMEOUT = 1u << 5;

// ------------------------------------------------------------------ formats
template <int FMT> struct Fmt;
template <> struct Fmt<4> {   // E2M1 (NVFP4 element)
  static constexpr int BLOCK_BYTES = 32;
  static constexpr float EMAX = 6.0f;
  static constexpr float DENOM = 2688.0f;     // maxB_ef * 448
  static constexpr uint32_t SBIT = 0x8, MAG = 0x7;
};
template <> struct Fmt<6> {   // E2M3 (6-bit element)
  static constexpr int BLOCK_BYTES = 48;
  static constexpr float EMAX = 7.5f;
  static constexpr float DENOM = 3360.0f;
  static constexpr uint32_t SBIT = 0x20, MAG = 0x1F;
};
template <> struct Fmt<8> {   // E4M3 element (8-bit variant)
  static constexpr int BLOCK_BYTES = 64;
  static constexpr float EMAX = 448.0f;
  static constexpr float DENOM = 200704.0f;
  static constexpr uint32_t SBIT = 0x80, MAG = 0x7F;
};

// max(a, b) that returns NaN when either is NaN (max.NaN.f32)
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// (a0 * b, a1 * b), each rounded to nearest even: one packed f32x2 multiply
__device__ __forceinline__ void mul2(float a0, float a1, float b, float &d0, float &d1) {
  uint64_t a, bb, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(bb) : "f"(b));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(bb));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

// Two fp32 -> two codes, round-to-nearest-even, saturating.  The returned
// value holds the code of `lo` in its low container (low nibble for E2M1,
// low byte for E2M3/E4M3) and the code of `hi` in the next one.
template <int FMT> __device__ __forceinline__ uint32_t cvt2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t cvt2<4>(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 q; cvt.rn.satfinite.e2m1x2.f32 q, %1, %2; cvt.u32.u8 %0, q; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
template <> __device__ __forceinline__ uint32_t cvt2<6>(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
template <> __device__ __forceinline__ uint32_t cvt2<8>(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two codes (low / high container as above) -> two exact fp16 values.
template <int FMT> __device__ __forceinline__ uint32_t dec2(uint32_t pair);
template <> __device__ __forceinline__ uint32_t dec2<4>(uint32_t pair) {
  uint32_t r;
  asm("{ .reg .b8 q; .reg .b16 w; cvt.u16.u32 w, %1; cvt.u8.u16 q, w; cvt.rn.f16x2.e2m1x2 %0, q; }"
      : "=r"(r) : "r"(pair));
  return r;
}
template <> __device__ __forceinline__ uint32_t dec2<6>(uint32_t pair) {
  uint32_t r;
  asm("{ .reg .b16 w; cvt.u16.u32 w, %1; cvt.rn.f16x2.e2m3x2 %0, w; }" : "=r"(r) : "r"(pair));
  return r;
}
template <> __device__ __forceinline__ uint32_t dec2<8>(uint32_t pair) {
  uint32_t r;
  asm("{ .reg .b16 w; cvt.u16.u32 w, %1; cvt.rn.f16x2.e4m3x2 %0, w; }" : "=r"(r) : "r"(pair));
  return r;
}

// magnitude value of one code of format FMT (exact)
template <int FMT> __device__ __forceinline__ float code_value(uint32_t mag) {
  uint32_t h = dec2<FMT>(mag);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Relative half-width of the bracket [q(1-eps), q(1+eps)] that is sure to
// contain the exact quotient when q is computed with a few fp32 roundings.
constexpr float QEPS = 9.5367431640625e-07f;   // 2^-20

// Tiny tensor scales.  The bracket and tie-test arguments below need
// B_scale * T_scale and maxB_ef * T_scale to be normal fp32 numbers, and the
// exact difference in the fma tie test to be a multiple of 2^-149.  Both hold
// for T_scale >= 2^-62 (the products are then >= 2^-71, and every term of the
// difference is a multiple of 2^-107 or finer than 2^-149 only below
// T_scale = 2^-107).  A tensor whose T_scale lies below 2^-62 (amax below
// about 1.2e-15) -- including a subnormal T_scale, amax below about 3e-35 --
// is encoded from x * 2^64 and T_scale * 2^64 instead: both products are exact
// powers-of-two shifts, so every quotient x / (B_scale * T_scale) is the same
// real number, and every intermediate is back in the range the arguments
// cover.  An input beyond 2^64 (only possible with a supplied statistic far
// below the data) would overflow; it is clamped to the largest finite value,
// whose quotient saturates all the same.
constexpr float TINY_ST = 0x1p-62f;
constexpr float TINY_MULT = 0x1p64f;
__device__ __forceinline__ bool is_tiny_scale(float s_t) { return s_t > 0.0f && s_t < TINY_ST; }
__device__ __forceinline__ float up64(float x) { return fminf(fmaxf(x * TINY_MULT, -3.4028234663852886e38f), 3.4028234663852886e38f); }

// Exact RN-even of the real quotient a / (k * s_t) onto the format grid, given
// the codes c_lo, c_hi of the bracket ends.  When they differ, the two are
// adjacent grid points and the one whose side of their midpoint `a` lies on
// is chosen; the comparison a <> mid * k * s_t is exact because mid * k is
// exact in fp32 (few significant bits) and fma rounds the exact difference
// once, which preserves its sign (and zero).  Inputs non-negative.
template <int FMT> __device__ __noinline__ uint32_t resolve_tie(float a, float k, float s_t, uint32_t c_lo,
                                                                 uint32_t c_hi) {
  uint32_t lo = c_lo < c_hi ? c_lo : c_hi, hi = c_lo < c_hi ? c_hi : c_lo;
  float mid = 0.5f * (code_value<FMT>(lo) + code_value<FMT>(hi));
  float r = fmaf(-(mid * k), s_t, a);
  if (r > 0.0f) return hi;
  if (r < 0.0f) return lo;
  return (lo & 1u) ? hi : lo;
}

// Block scale code: RN_E4M3(amax_b / (maxB_ef * s_t)), satfinite, exact.
template <int FMT> __device__ __forceinline__ uint32_t block_scale_code(float amax_b, float s_t) {
  if (!(s_t > 0.0f)) return 0u;
  float q = __fdiv_rn(amax_b, Fmt<FMT>::EMAX * s_t);
  uint32_t c_lo = cvt2<8>(q * (1.0f - QEPS), 0.0f) & 0xFFu;
  uint32_t c_hi = cvt2<8>(q * (1.0f + QEPS), 0.0f) & 0xFFu;
  if (c_lo == c_hi) return c_lo;
  return resolve_tie<8>(amax_b, Fmt<FMT>::EMAX, s_t, c_lo, c_hi);
}

// Same decision as block_scale_code, with the quotient formed from a
// precomputed inv_den = rcp(maxB_ef * s_t): the bracket [q(1-eps), q(1+eps)]
// still contains the exact quotient (a few fp32 roundings, each 2^-24, are
// far inside eps = 2^-20) and the tie test stays exact.
template <int FMT>
__device__ __forceinline__ uint32_t block_scale_code_r(float amax_b, float s_t, float inv_den) {
  if (!(s_t > 0.0f)) return 0u;
  const float q = amax_b * inv_den;
  uint32_t c_lo = cvt2<8>(q * (1.0f - QEPS), 0.0f) & 0xFFu;
  uint32_t c_hi = cvt2<8>(q * (1.0f + QEPS), 0.0f) & 0xFFu;
  if (c_lo == c_hi) return c_lo;
  return resolve_tie<8>(amax_b, Fmt<FMT>::EMAX, s_t, c_lo, c_hi);
}

// ------------------------------------------------------------- misc device
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `sleep_ns` inside the
// instruction; it wakes as soon as the phase completes.  Long hints keep
// waiting warps from re-polling shared memory.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t sleep_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(sleep_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// `limit_ns` of wall time, sets ST_TIMEOUT in *status and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, ST_TIMEOUT);
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// whole warp: allocate `ncols` TMEM columns (power of two >= 32), address -> *slot
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// Shared-memory matrix descriptor, no swizzle.  lbo: byte distance between
// core matrices adjacent along K; sbo: along M/N.  Bits 46-48 = 0b001.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// a shared-memory descriptor from its two 32-bit words
__device__ __forceinline__ uint64_t desc_of(uint32_t hi, uint32_t lo) { return ((uint64_t)hi << 32) | lo; }

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// the same, always accumulating into D
__device__ __forceinline__ void umma_f16_acc(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{ .reg .pred p; setp.eq.u32 p, 0, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc));
}
// arrive on `bar` once every tcgen05 op issued so far by this thread completed
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 32 bits, 32 consecutive columns per thread
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace mq

namespace mq {

// ------------------------------------------------------------------- TMA
// arrive once on `bar` and add `bytes` to the transaction count it waits for
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// tiled tensor loads (global -> this CTA's shared memory); completion is
// signalled on `bar` as transaction bytes.  Out-of-range boxes read zeros.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(void *dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2,
                                            int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

}  // namespace mq

namespace mq {

// ------------------------------------------------------------ block decode
// Row `r` (eight consecutive in-block elements 8r .. 8r+7) of a packed block
// is fetched raw (load_raw) and turned into eight fp16 values code * scale
// (decode_raw, 16 bytes).  `s2` holds the block scale in both halves of an
// f16x2 (already multiplied by the operand pre-scale).
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  __half2 x = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&x);
}

template <int F> __device__ __forceinline__ uint4 decode_raw(uint2 w, uint32_t s2) {
  if (F == 4) {
    return make_uint4(hmul2u(dec2<4>(w.x), s2), hmul2u(dec2<4>(w.x >> 8), s2), hmul2u(dec2<4>(w.x >> 16), s2),
                      hmul2u(dec2<4>(w.x >> 24), s2));
  } else if (F == 8) {
    return make_uint4(hmul2u(dec2<8>(w.x), s2), hmul2u(dec2<8>(w.x >> 16), s2), hmul2u(dec2<8>(w.y), s2),
                      hmul2u(dec2<8>(w.y >> 16), s2));
  } else {
    const uint64_t v = (uint64_t)w.x | ((uint64_t)w.y << 32);   // 8 x 6-bit codes, element j at bits 6j
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = (uint32_t)(v >> (12 * k)) & 0x3Fu, hi = (uint32_t)(v >> (12 * k + 6)) & 0x3Fu;
      q[k] = hmul2u(dec2<6>(lo | (hi << 8)), s2);
    }
    return make_uint4(q[0], q[1], q[2], q[3]);
  }
}

// raw bits of row r (8 codes) of a packed block (shared or global memory,
// 16-byte aligned)
template <int F> __device__ __forceinline__ uint2 row8_bits(const uint8_t *blk, int r) {
  if (F == 4) return make_uint2(*reinterpret_cast<const uint32_t *>(blk + 4 * r), 0u);
  if (F == 8) return *reinterpret_cast<const uint2 *>(blk + 8 * r);
  // E2M3: row r is bytes 6r .. 6r+5 of the 48-byte block; two aligned 32-bit
  // loads from byte 6r rounded down to a multiple of 4 (at most byte 47
  // read) and a funnel shift by 0 or 16 bits
  const uint32_t *w = reinterpret_cast<const uint32_t *>(blk + ((6 * r) & ~3));
  const uint32_t w0 = w[0], w1 = w[1], sh = (uint32_t)((6 * r) & 2) * 8u;
  return make_uint2(__funnelshift_r(w0, w1, sh), (w1 >> sh) & 0xFFFFu);
}

// fp16 pair holding the E4M3 block scale (times 1/4 for E4M3-coded operands,
// whose code * scale can exceed the fp16 range; the epilogue multiplies back).
template <int F> __device__ __forceinline__ uint32_t scale_pair(uint8_t sc) {
  uint32_t h = dec2<8>((uint32_t)sc) & 0xFFFFu;
  if (F == 8) h = hmul2u(h, 0x3400u);   // x 0.25 (exact: a power of two, stays normal)
  return h | (h << 16);
}

}  // namespace mq

namespace mq {

// -------------------------------------------------------------- cp.async
// Asynchronous global -> shared copy of BYTES (4, 8 or 16) bytes; when
// `valid` is false nothing is read and the destination is zero-filled.
template <int BYTES>
__device__ __forceinline__ void cp_async_zfill(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(smem_u32(dst)), "l"(src), "n"(BYTES),
               "r"(valid ? BYTES : 0)
               : "memory");
}
// arrive on `bar` once every cp.async this thread issued so far has landed
// (counts as one of the barrier's expected arrivals)
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// add `bytes` to the transaction count of the current phase without arriving
__device__ __forceinline__ void mbar_add_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Copy `nruns` byte runs into shared memory: run r has `len(r)` valid bytes
// (a multiple of GRAN) starting at `src(r)` (GRAN-aligned; null: no valid
// bytes) and occupies `fill` bytes at dst + r * stride, the bytes past
// len(r) zero-filled.  Lane-strided over a warp.  GRAN >= 4 issues cp.async
// copies (complete them with cp_async_arrive); GRAN 1 or 2 copies
// synchronously (complete with an ordinary arrive).
template <int GRAN, class SrcF, class LenF>
__device__ __forceinline__ void copy_runs(uint8_t *dst, int nruns, int stride, int fill, SrcF src, LenF len,
                                          const uint8_t *safe, int lane) {
  const int per = fill / GRAN;
  for (int i = lane; i < nruns * per; i += 32) {
    const int r = i / per, part = i - r * per;
    const uint8_t *s = src(r);
    const bool ok = s != nullptr && part * GRAN < len(r);
    uint8_t *d = dst + r * stride + part * GRAN;
    if constexpr (GRAN >= 4) {
      cp_async_zfill<GRAN>(d, ok ? s + part * GRAN : safe, ok);
    } else {
      uint8_t v[GRAN];
#pragma unroll
      for (int b = 0; b < GRAN; ++b) v[b] = ok ? __ldg(s + part * GRAN + b) : (uint8_t)0;
#pragma unroll
      for (int b = 0; b < GRAN; ++b) d[b] = v[b];
    }
  }
}

// copy_runs with the granule chosen at run time (1, 2, 4, 8 or 16).  A
// stage filled this way completes with two arrivals per lane:
// cp_async_arrive (the asynchronous copies) and mbar_arrive (release of the
// synchronous ones).
// `safe`: any valid global address, given to zero-filling copies that read nothing.
template <class SrcF, class LenF>
__device__ __forceinline__ void copy_runs_rt(int gran, uint8_t *dst, int nruns, int stride, int fill, SrcF src,
                                             LenF len, const uint8_t *safe, int lane) {
  switch (gran) {
    case 16: copy_runs<16>(dst, nruns, stride, fill, src, len, safe, lane); break;
    case 8: copy_runs<8>(dst, nruns, stride, fill, src, len, safe, lane); break;
    case 4: copy_runs<4>(dst, nruns, stride, fill, src, len, safe, lane); break;
    case 2: copy_runs<2>(dst, nruns, stride, fill, src, len, safe, lane); break;
    default: copy_runs<1>(dst, nruns, stride, fill, src, len, safe, lane); break;
  }
}

}  // namespace mq

namespace mq {

// Codes of eight fp32 values (one block row) for block scale value bs and
// T_scale s_t (encode_row8 / encode_row8_b below): exact RN of the real
// quotient x / (bs * s_t), from the bracket and the fma-sign test of
// tie_quotient.  Returns the packed row: element j at bits 4j (E2M1), 6j
// (E2M3) or 8j (E4M3).
//
// Bracket multipliers of the quotient x / (bs * s_t) (0 when bs is 0).  The
// reciprocal is the hardware approximation (relative error below 2^-22);
// with the product bs * s_t and the three later roundings (each 2^-24) the
// computed ends still lie below and above the exact quotient, since the
// bracket half-width is 2^-20.
__device__ __forceinline__ void quot_bracket(float bs, float s_t, float &inv_lo, float &inv_hi) {
  inv_lo = inv_hi = 0.0f;
  if (bs > 0.0f) {
    float inv;
    asm("rcp.approx.f32 %0, %1;" : "=f"(inv) : "f"(bs * s_t));
    inv_lo = inv * (1.0f - QEPS);
    inv_hi = inv * (1.0f + QEPS);
  }
}

template <int F>
__device__ __forceinline__ uint64_t encode_row8_b(const float (&v)[8], float bs, float s_t, float inv_lo, float inv_hi);

template <int F> __device__ __forceinline__ uint64_t encode_row8(const float (&v)[8], float bs, float s_t) {
  float inv_lo, inv_hi;
  quot_bracket(bs, s_t, inv_lo, inv_hi);
  return encode_row8_b<F>(v, bs, s_t, inv_lo, inv_hi);
}

// encode_row8 with the bracket multipliers of quot_bracket precomputed.  The
// codes of both bracket ends are formed for the whole row at once; when they
// agree (the common case) the row is placed as is, otherwise every element is
// converted again from the quotient tie_quotient picks, without a branch.
//
// tie_quotient: a value whose RN-even conversion is the exact RN-even code of
// the quotient x / (bs * s_t), given the bracket ends ql, qh around it
// (signed like x; |ql| <= |qh|).  m = ql rounded to 5 significant bits is the
// rounding midpoint inside the bracket when there is one: every midpoint of
// the three grids has at most 5 significant bits, and the bracket is 2^-19
// wide.  The fma rounds the exact |x| - (|m| * bs) * s_t once (|m| * bs is
// exact: at most 9 significant bits), so its sign is the side of m on which
// the exact quotient lies (the argument of resolve_tie): above m the code of
// qh is right, below it the code of ql, and on it the exact quotient is m
// itself, which the conversion rounds to even.  Without a midpoint in the
// bracket both ends convert to the same code, and so does m when the sign is
// zero (m is then the exact quotient).
__device__ __forceinline__ float tie_quotient(float ql, float qh, float x, float bs, float s_t) {
  const float m = __uint_as_float((__float_as_uint(ql) + 0x40000u) & 0xFFF80000u);
  const float r = fmaf(-(fabsf(m) * bs), s_t, fabsf(x));
  return r > 0.0f ? qh : (r < 0.0f ? ql : m);
}

// E2M3 codes in byte containers (element j in byte j, the code in its low
// 6 bits) -> the packed 6-bit row (element j at bits 6j): four codes of a
// 32-bit half are compacted in two shift-and-mask steps (pairs into 12-bit
// fields, then the two fields into 24 bits)
__device__ __forceinline__ uint32_t compact_e2m3x4(uint32_t x) {
  x = (x & 0x003F003Fu) | ((x >> 2) & 0x0FC00FC0u);
  return (x & 0x00000FFFu) | ((x >> 4) & 0x00FFF000u);
}
__device__ __forceinline__ uint64_t pack_e2m3_row(uint64_t b) {
  return (uint64_t)compact_e2m3x4((uint32_t)b) | ((uint64_t)compact_e2m3x4((uint32_t)(b >> 32)) << 24);
}

// eight quotients -> one row of codes in containers (E2M1: nibbles, E2M3 /
// E4M3: bytes, element j in container j); E2M1: four
// byte pairs packed in one step, E4M3: four 16-bit pairs
__device__ __forceinline__ uint32_t cvt_row_e2m1(const float (&q)[8]) {
  uint32_t r;
  asm("{ .reg .b8 a, b, c, d;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 a, %2, %1;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b, %4, %3;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 c, %6, %5;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 d, %8, %7;\n"
      "  mov.b32 %0, {a, b, c, d}; }"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}
__device__ __forceinline__ uint64_t cvt_row_e4m3(const float (&q)[8]) {
  uint64_t r;
  asm("{ .reg .b16 a, b, c, d;\n"
      "  cvt.rn.satfinite.e4m3x2.f32 a, %2, %1;\n"
      "  cvt.rn.satfinite.e4m3x2.f32 b, %4, %3;\n"
      "  cvt.rn.satfinite.e4m3x2.f32 c, %6, %5;\n"
      "  cvt.rn.satfinite.e4m3x2.f32 d, %8, %7;\n"
      "  mov.b64 %0, {a, b, c, d}; }"
      : "=l"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

__device__ __forceinline__ uint64_t cvt_row_e2m3(const float (&q)[8]) {
  uint64_t r;
  asm("{ .reg .b16 a, b, c, d;\n"
      "  cvt.rn.satfinite.e2m3x2.f32 a, %2, %1;\n"
      "  cvt.rn.satfinite.e2m3x2.f32 b, %4, %3;\n"
      "  cvt.rn.satfinite.e2m3x2.f32 c, %6, %5;\n"
      "  cvt.rn.satfinite.e2m3x2.f32 d, %8, %7;\n"
      "  mov.b64 %0, {a, b, c, d}; }"
      : "=l"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

template <int F>
__device__ __forceinline__ uint64_t encode_row8_b(const float (&v)[8], float bs, float s_t, float inv_lo, float inv_hi) {
  float ql[8], qh[8];
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    mul2(v[2 * jj], v[2 * jj + 1], inv_lo, ql[2 * jj], ql[2 * jj + 1]);
    mul2(v[2 * jj], v[2 * jj + 1], inv_hi, qh[2 * jj], qh[2 * jj + 1]);
  }
  // whole rows at once (codes in nibble / byte containers), compared once
  const uint64_t row_lo = F == 4 ? (uint64_t)cvt_row_e2m1(ql) : F == 8 ? cvt_row_e4m3(ql) : cvt_row_e2m3(ql);
  const uint64_t row_hi = F == 4 ? (uint64_t)cvt_row_e2m1(qh) : F == 8 ? cvt_row_e4m3(qh) : cvt_row_e2m3(qh);
  uint64_t row = row_lo;
  if (row_lo != row_hi) {   // some element near a midpoint: convert the row again from the picked quotients
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = tie_quotient(ql[j], qh[j], v[j], bs, s_t);
    row = F == 4 ? (uint64_t)cvt_row_e2m1(q) : F == 8 ? cvt_row_e4m3(q) : cvt_row_e2m3(q);
  }
  if constexpr (F == 6) return pack_e2m3_row(row);
  return row;
}

// store one packed row (8 codes) at byte offset 4r / 6r / 8r of its block
template <int F> __device__ __forceinline__ void store_row8(uint8_t *blk, int r, uint64_t bits) {
  if (F == 4) {
    reinterpret_cast<uint32_t *>(blk)[r] = (uint32_t)bits;
  } else if (F == 6) {
    uint16_t *d16 = reinterpret_cast<uint16_t *>(blk + 6 * r);
    d16[0] = (uint16_t)bits;
    d16[1] = (uint16_t)(bits >> 16);
    d16[2] = (uint16_t)(bits >> 32);
  } else {
    reinterpret_cast<uint64_t *>(blk)[r] = bits;
  }
}

}  // namespace mq

namespace mq {

// ------------------------------------------------------ stochastic rounding
// MicroQonv §III-A lets Round be stochastic (the paper's choice for
// gradients).  Random words come from Philox4x32-10 (Salmon, Moraes, Dror,
// Shaw, SC 2011) keyed by a 64-bit seed; element e of a packed tensor
// (e = block * 64 + in-block index) takes word e % 4 of counter
// (e / 4 low, e / 4 high, 0, 0).  The decision is taken in fp32, exactly at
// every step: q = fl32(|x| / fl32(B_scale T_scale)) (IEEE division, so
// subnormal and tiny scales need no rescaling here); q >= maxB_ef gives the
// largest code; otherwise, with lo <= q < hi the grid values around q, the
// code is hi when (top 24 bits of the word) < 2^24 (q - lo) / (hi - lo).
// q - lo is exact (lo <= q <= 2 lo, or lo = 0) and hi - lo is a power of two.

// Philox4x32-10 of counter c (in place) under key (k0, k1)
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
    const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// stochastic magnitude code of ax = |x| >= 0 for d = fl32(B_scale T_scale)
template <int F> __device__ __forceinline__ uint32_t sr_mag(float ax, float d, uint32_t word) {
  const float q = __fdiv_rn(ax, d);
  if (!(q > 0.0f)) return 0u;
  constexpr uint32_t MAXC = F == 8 ? 0x7Eu : Fmt<F>::MAG;   // largest finite magnitude code
  if (q >= Fmt<F>::EMAX) return MAXC;
  const uint32_t c = cvt2<F>(q, 0.0f) & Fmt<F>::MAG;        // nearest grid value (q below the largest)
  const uint32_t lo = code_value<F>(c) > q ? c - 1u : c;
  const float g_lo = code_value<F>(lo), g_hi = code_value<F>(lo + 1u);
  const float frac = __fmul_rn(__fsub_rn(q, g_lo), __frcp_rn(__fsub_rn(g_hi, g_lo)));   // exact
  const float scaled = __fmul_rn(frac, 16777216.0f);
  return __uint2float_rn(word >> 8) < scaled ? lo + 1u : lo;
}

// Codes of one block row v[0..7] (elements 8r .. 8r+7 of block blk), packed
// like encode_row8's result; d = fl32(B_scale T_scale), 0 for a zero scale.
template <int F>
__device__ __forceinline__ uint64_t encode_row8_sr(const float (&v)[8], float d, uint64_t seed, int64_t blk, int r) {
  uint64_t bits = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t ctr = (uint64_t)blk * 16u + (uint64_t)(2 * r + h);   // element index / 4
    uint32_t w[4] = {(uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u};
    philox4x32_10(w, (uint32_t)seed, (uint32_t)(seed >> 32));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x = v[4 * h + j];
      const uint32_t mag = d > 0.0f ? sr_mag<F>(fabsf(x), d, w[j]) : 0u;
      const uint32_t code = mag | (signbit(x) ? Fmt<F>::SBIT : 0u);
      bits |= (uint64_t)code << ((F == 4 ? 4 : F == 6 ? 6 : 8) * (4 * h + j));
    }
  }
  return bits;
}

}  // namespace mq
