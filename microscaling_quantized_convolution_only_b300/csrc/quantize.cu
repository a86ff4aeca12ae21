// quantize.cu -- quantize a dense tensor once into packed square 8x8 blocks.
//
// MicroQonv §III-A / §IV-B: T_scale = amax / (maxB_ef * 448); per 8x8 block
// B_scale = CastE4M3(amax_block / (maxB_ef * T_scale)); codes
// Round(x / (B_scale * T_scale)).  Blocks span (N, C_in) for activations,
// (C_out, C_in) for weights and (N, C_out) for output gradients and are stored
// channel-batch-first (§IV-A): block order [H][W][N/8][C/8], element i = 8n + c.
//
// One thread owns one block: it gathers the block's 64 inputs (for NCHW
// inputs consecutive lanes own consecutive spatial positions, so each of the
// 64 loads is a coalesced warp-wide row segment, from a TMA-filled shared
// stage or straight from global memory; for HWCN inputs each lane reads eight
// 8-element rows), reduces the block amax in registers, derives the E4M3
// block scale exactly, converts the codes with the hardware RN conversions on
// a bracket [q(1-eps), q(1+eps)] of the quotient and settles a row whose
// bracket straddles a rounding midpoint with an exact fma-sign test
// (tie_quotient).  Codes and the scale byte are written once, straight to
// their place in global memory.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace mq {

__device__ __forceinline__ float load_elem(const float *p) { return __ldg(p); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }

// ------------------------------------------------------------------ amax
// max |x| over a flat array; the fp32 bit patterns of |x| order like the
// values (Inf and NaN above every finite value), so an unsigned max works.
template <typename T>
__global__ void __launch_bounds__(256) amax_kernel(const T *__restrict__ src, int64_t n, uint32_t *amax_bits) {
  uint32_t m = 0;
  constexpr int V = 16 / sizeof(T);
  int64_t nv = n / V;
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv; i += (int64_t)gridDim.x * blockDim.x) {
    uint4 v = __ldg(s4 + i);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (sizeof(T) == 4) {
        m = max(m, w[j] & 0x7FFFFFFFu);
      } else {
        m = max(m, (w[j] << 16) & 0x7FFFFFFFu);
        m = max(m, w[j] & 0x7FFF0000u);
      }
    }
  }
  for (int64_t i = nv * V + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    m = max(m, __float_as_uint(fabsf(load_elem(src + i))));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (threadIdx.x == 0 && m) atomicMax(amax_bits, m);
  }
}

// ------------------------------------------------------------- codes
// Row sink of the block encoders: the packed rows of one block collected in
// registers and written to the block's place in global memory with 32- or
// 16-byte stores (block payload layout in mqconv.h).
template <int F> struct RegRows {
  static constexpr int NW = Fmt<F>::BLOCK_BYTES / 4;
  uint32_t w[NW];
  // r is a constant after unrolling; E2M3 rows are 48 bits, so an odd row
  // starts in the upper half of a word that the row before it began
  __device__ __forceinline__ void put(int r, uint64_t bits) {
    if (F == 4) {
      w[r] = (uint32_t)bits;
    } else if (F == 8) {
      w[2 * r] = (uint32_t)bits;
      w[2 * r + 1] = (uint32_t)(bits >> 32);
    } else if ((r & 1) == 0) {
      w[3 * r / 2] = (uint32_t)bits;
      w[3 * r / 2 + 1] = (uint32_t)(bits >> 32);
    } else {
      w[(3 * r - 1) / 2] |= (uint32_t)bits << 16;
      w[(3 * r + 1) / 2] = (uint32_t)(bits >> 16);
    }
  }
  // 32-byte stores where the payload starts on a 32-byte boundary (every
  // sector written whole in one request), else 16-byte stores
  __device__ __forceinline__ void st32(uint8_t *d, int k) const {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d), "r"(w[k]), "r"(w[k + 1]),
                 "r"(w[k + 2]), "r"(w[k + 3]), "r"(w[k + 4]), "r"(w[k + 5]), "r"(w[k + 6]), "r"(w[k + 7])
                 : "memory");
  }
  __device__ __forceinline__ void st16(uint8_t *d, int k) const {
    *reinterpret_cast<uint4 *>(d) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
  }
  __device__ __forceinline__ void store(uint8_t *dst) const {
    const bool a32 = (reinterpret_cast<uintptr_t>(dst) & 31u) == 0;
    if (F == 6) {                                  // 48 bytes: 32 + 16 or 16 + 32
      if (a32) {
        st32(dst, 0);
        st16(dst + 32, 8);
      } else {
        st16(dst, 0);
        st32(dst + 16, 4);
      }
    } else if (a32) {
#pragma unroll
      for (int k = 0; k < NW / 8; ++k) st32(dst + 32 * k, 8 * k);
    } else {
#pragma unroll
      for (int k = 0; k < NW / 4; ++k) st16(dst + 16 * k, 4 * k);
    }
  }
};

// -------------------------------------------------------------- quantize
// Thread order: NCHW/OIHW -- spatial position fastest; HWCN -- n-group fastest.
template <int FMT, typename T, int LAYOUT, bool SR>
__global__ void __launch_bounds__(256) quantize_kernel(const T *__restrict__ src, QuantParams p) {
  const int64_t GA = p.d0 / 8, GB = p.d1 / 8, HW = p.d2 * p.d3;
  const int64_t nblk = GA * GB * HW;
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;

  // T_scale from the statistic (identical in every thread: one fp32 division)
  const float amax_src = __uint_as_float(*p.amax_src_bits);
  const float s_t = __fdiv_rn(amax_src, Fmt<FMT>::DENOM);
  if (t == 0) {
    *p.s_t_out = s_t;
    if (!(amax_src <= 3.4028234663852886e38f)) atomicOr(p.status, ST_NONFINITE);
  }

  uint32_t my_amax = 0;
  if (t < nblk) {
    int64_t hw, ga, gb;
    if (LAYOUT == 1) {   // HWCN
      ga = t % GA;
      gb = (t / GA) % GB;
      hw = t / (GA * GB);
    } else {
      hw = t % HW;
      gb = (t / HW) % GB;
      ga = t / (HW * GB);
    }
    float x[64];
    if (LAYOUT == 1) {
      // [H][W][C][N]: row c holds 8 contiguous n
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const T *row = src + ((hw * p.d1 + gb * 8 + c) * p.d0 + ga * 8);
        if (sizeof(T) == 4) {
          const float4 a = __ldg(reinterpret_cast<const float4 *>(row));
          const float4 b = __ldg(reinterpret_cast<const float4 *>(row) + 1);
          x[0 * 8 + c] = a.x; x[1 * 8 + c] = a.y; x[2 * 8 + c] = a.z; x[3 * 8 + c] = a.w;
          x[4 * 8 + c] = b.x; x[5 * 8 + c] = b.y; x[6 * 8 + c] = b.z; x[7 * 8 + c] = b.w;
        } else {
          const uint4 a = __ldg(reinterpret_cast<const uint4 *>(row));
          const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            x[(2 * k) * 8 + c] = __uint_as_float(w[k] << 16);
            x[(2 * k + 1) * 8 + c] = __uint_as_float(w[k] & 0xFFFF0000u);
          }
        }
      }
    } else {
      // NCHW / OIHW: element (a, b) at ((a * d1 + b) * HW + hw)
      const T *base = src + ((ga * 8) * p.d1 + gb * 8) * HW + hw;
#pragma unroll
      for (int i = 0; i < 64; ++i) x[i] = load_elem(base + ((i >> 3) * p.d1 + (i & 7)) * HW);
    }
    // |x| bit patterns order like the values, with Inf and NaN above all finite ones
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 64; ++i) mb = max(mb, __float_as_uint(x[i]) & 0x7FFFFFFFu);
    my_amax = mb;
    if (mb >= 0x7F800000u) atomicOr(p.status, ST_NONFINITE);
    float amax_b = __uint_as_float(mb);
    const int64_t b = (hw * GA + ga) * GB + gb;
    if (SR) {   // stochastic element codes (the block scale is round-to-nearest)
      const uint32_t bs_code = is_tiny_scale(s_t) ? block_scale_code<FMT>(up64(amax_b), s_t * TINY_MULT)
                                                  : block_scale_code<FMT>(amax_b, s_t);
      const float d = __fmul_rn(code_value<8>(bs_code), s_t);
      uint8_t *blkp = p.codes + b * Fmt<FMT>::BLOCK_BYTES;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = x[8 * r + c];
        store_row8<FMT>(blkp, r, encode_row8_sr<FMT>(v, d, p.sr_seed, b, r));
      }
      p.scales[b] = (uint8_t)bs_code;
    } else {
      float st = s_t;
      if (is_tiny_scale(s_t)) {   // T_scale below 2^-62: encode from x 2^64, T_scale 2^64 (see up64)
        st = s_t * TINY_MULT;
        amax_b = up64(amax_b);
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = up64(x[i]);
      }
      const uint32_t bs_code = block_scale_code<FMT>(amax_b, st);
      const float bs = code_value<8>(bs_code);
      float inv_lo, inv_hi;
      quot_bracket(bs, st, inv_lo, inv_hi);
      RegRows<FMT> rows;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = x[8 * r + c];
        rows.put(r, encode_row8_b<FMT>(v, bs, st, inv_lo, inv_hi));
      }
      rows.store(p.codes + b * Fmt<FMT>::BLOCK_BYTES);
      p.scales[b] = (uint8_t)bs_code;
    }
  }

  if (p.amax_meas_bits) {
    uint32_t m = my_amax;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0 && m) atomicMax(p.amax_meas_bits, m);
  }
}


// raw input bits (bf16 zero-extended) and their fp32 bit pattern
__device__ __forceinline__ uint32_t load_bits(const float *p) { return __float_as_uint(__ldg(p)); }
__device__ __forceinline__ uint32_t load_bits(const __nv_bfloat16 *p) {
  return (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p));
}
template <typename T> __device__ __forceinline__ uint32_t to_bits32(uint32_t raw) {
  return sizeof(T) == 2 ? raw << 16 : raw;
}

// Block scale and codes of one block whose 64 inputs are held as raw bits
// (bf16 inputs two to a register, element 2k in the low half), row a of the
// block (8 consecutive b) at raw[8a / PK ...]; `mb` is the block amax (fp32
// bits).  The packed rows go to the sink `ob` (a RegRows); returns
// the E4M3 scale code.  TINY:
// T_scale below 2^-62, encoded from x 2^64 and T_scale 2^64 (see up64).
// inv_den: block_den_rcp<FMT, TINY>(s_t), the reciprocal the block-scale
// quotient is formed with (the same for every block; the bracket test keeps
// the decision exact).
template <int FMT, bool TINY> __device__ __forceinline__ float block_den_rcp(float s_t) {
  return __frcp_rn(Fmt<FMT>::EMAX * (TINY ? s_t * TINY_MULT : s_t));
}

template <int FMT, typename T, bool TINY, class Sink>
__device__ __forceinline__ uint32_t encode_raw_block(const uint32_t (&raw)[sizeof(T) == 2 ? 32 : 64], uint32_t mb,
                                                     float s_t, float inv_den, Sink &ob) {
  const float st = TINY ? s_t * TINY_MULT : s_t;
  const float amax_b = TINY ? up64(__uint_as_float(mb)) : __uint_as_float(mb);
  const uint32_t bs_code = block_scale_code_r<FMT>(amax_b, st, inv_den);
  const float bs = code_value<8>(bs_code);
  float inv_lo, inv_hi;
  quot_bracket(bs, st, inv_lo, inv_hi);
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    float x[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (sizeof(T) == 2) {
        const uint32_t w = raw[((a * 8 + b) / 2) & 31];
        x[b] = __uint_as_float((b & 1) ? (w & 0xFFFF0000u) : (w << 16));
      } else {
        x[b] = __uint_as_float(raw[(a * 8 + b) & 63]);
      }
      if (TINY) x[b] = up64(x[b]);
    }
    ob.put(a, encode_row8_b<FMT>(x, bs, st, inv_lo, inv_hi));
  }
  return bs_code;
}

// The same block with stochastically rounded element codes (block `blk` of
// the packed tensor, Philox key `seed`; see encode_row8_sr).  The block scale
// is the round-to-nearest one.
template <int FMT, typename T, class Sink>
__device__ __forceinline__ uint32_t encode_raw_block_sr(const uint32_t (&raw)[sizeof(T) == 2 ? 32 : 64], uint32_t mb,
                                                        float s_t, Sink &ob, int64_t blk, uint64_t seed) {
  const bool tiny = is_tiny_scale(s_t);
  const float amax_b = __uint_as_float(mb);
  const uint32_t bs_code = tiny ? block_scale_code<FMT>(up64(amax_b), s_t * TINY_MULT)
                                : block_scale_code<FMT>(amax_b, s_t);
  const float d = __fmul_rn(code_value<8>(bs_code), s_t);
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    float x[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (sizeof(T) == 2) {
        const uint32_t w = raw[((a * 8 + b) / 2) & 31];
        x[b] = __uint_as_float((b & 1) ? (w & 0xFFFF0000u) : (w << 16));
      } else {
        x[b] = __uint_as_float(raw[(a * 8 + b) & 63]);
      }
    }
    ob.put(a, encode_row8_sr<FMT>(x, d, seed, blk, a));
  }
  return bs_code;
}

// ------------------------------------------------------ NCHW / OIHW path
// Dense NCHW (or OIHW: a = Cout, b = Cin, hw = tap) input is contiguous along
// hw; the packed output is contiguous along the b-groups of one (hw, a-group).
// A CTA of 8 warps takes one a-group, 8 b-groups (one per warp) and 32
// positions (one per lane): each thread quantizes one block from 64 loads that
// are coalesced across the warp (consecutive positions) and writes the packed
// block and its scale straight to global memory; the eight warps write
// neighbouring blocks, so lines fill in L2 before they are written back.
constexpr int QN_HW = 32, QN_GB = 8;

// CTA shape: GBT b-groups (one warp each) x (8 / GBT) chunks of 32 positions;
// GBT = min(8, B / 8) so that narrow tensors keep all warps busy.
// The work of one quantize_nchw_kernel CTA after T_scale is known (TINY:
// T_scale below 2^-62).
template <int FMT, typename T, bool SR, bool TINY>
__device__ __forceinline__ void nchw_body(const T *__restrict__ src, const QuantParams &p, float s_t) {
  constexpr int BB = Fmt<FMT>::BLOCK_BYTES;
  const int GA = (int)(p.d0 / 8), GB = (int)(p.d1 / 8);
  const int GBT = GB < QN_GB ? GB : QN_GB, HWT = QN_HW * (QN_GB / GBT);
  const int64_t HW = p.d2 * p.d3;
  const int64_t hw_tiles = (HW + HWT - 1) / HWT;
  const int gb_tiles = (GB + GBT - 1) / GBT;
  int64_t r = blockIdx.x;
  const int64_t hw0 = (r % hw_tiles) * HWT;
  r /= hw_tiles;
  const int gb0 = (int)(r % gb_tiles) * GBT;
  const int ga = (int)(r / gb_tiles);
  const int ngb = min(GBT, GB - gb0);
  const int nhw = (int)(HW - hw0 < (int64_t)HWT ? HW - hw0 : (int64_t)HWT);
  const int warp = threadIdx.x >> 5;
  const int wl = warp % GBT, hl = (warp / GBT) * 32 + (threadIdx.x & 31);
  uint32_t my_amax = 0;
  if (wl < ngb && hl < nhw) {
    // the block's 64 inputs, row a = 8 consecutive b; rows and columns are
    // HW elements apart, addressed by pointer increments
    const T *row = src + ((int64_t)(ga * 8) * p.d1 + (gb0 + wl) * 8) * HW + hw0 + hl;
    const int64_t rstride = p.d1 * HW;
    // values held as fp32 bit patterns; bf16 inputs two per register
    constexpr int PK = sizeof(T) == 2 ? 2 : 1;
    uint32_t raw[64 / PK];
#pragma unroll
    for (int a = 0; a < 8; ++a, row += rstride) {
      const T *q = row;
#pragma unroll
      for (int b = 0; b < 8; b += PK, q += PK * HW) {
        if (PK == 2) raw[(a * 8 + b) / 2] = load_bits(q) | (load_bits(q + HW) << 16);
        else raw[a * 8 + b] = load_bits(q);
      }
    }
    uint32_t mb = 0;
    if (PK == 2) {
      uint32_t m2 = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) m2 = __vmaxu2(m2, raw[i] & 0x7FFF7FFFu);
      mb = max(m2 << 16, m2 & 0xFFFF0000u);
    } else {
#pragma unroll
      for (int i = 0; i < 64 / PK; ++i) mb = max(mb, raw[i] & 0x7FFFFFFFu);
    }
    my_amax = mb;
    if (mb >= 0x7F800000u) atomicOr(p.status, ST_NONFINITE);
    const int64_t blk = ((hw0 + hl) * GA + ga) * (int64_t)GB + gb0 + wl;
    RegRows<FMT> rows;
    const uint32_t bs_code = SR ? encode_raw_block_sr<FMT, T>(raw, mb, s_t, rows, blk, p.sr_seed)
                                : encode_raw_block<FMT, T, TINY>(raw, mb, s_t, block_den_rcp<FMT, TINY>(s_t), rows);
    rows.store(p.codes + blk * BB);
    p.scales[blk] = (uint8_t)bs_code;
  }
  if (p.amax_meas_bits) {
    uint32_t m = my_amax;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0 && m) atomicMax(p.amax_meas_bits, m);
  }
}

template <int FMT, typename T>
__device__ __noinline__ void nchw_body_tiny(const T *__restrict__ src, const QuantParams &p, float s_t) {
  nchw_body<FMT, T, false, true>(src, p, s_t);
}

template <int FMT, typename T, bool SR>
__global__ void __launch_bounds__(256, 2) quantize_nchw_kernel(const T *__restrict__ src, QuantParams p) {
  const float amax_src = __uint_as_float(*p.amax_src_bits);
  const float s_t = __fdiv_rn(amax_src, Fmt<FMT>::DENOM);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *p.s_t_out = s_t;
    if (!(amax_src <= 3.4028234663852886e38f)) atomicOr(p.status, ST_NONFINITE);
  }
  // stochastic codes decide from the unscaled T_scale; the tiny-T_scale
  // round-to-nearest encode runs in an out-of-line copy
  if (!SR && is_tiny_scale(s_t)) nchw_body_tiny<FMT, T>(src, p, s_t);
  else nchw_body<FMT, T, SR, false>(src, p, s_t);
}


// ------------------------------------------------- NCHW / OIHW, TMA path
// Same tiling and arithmetic as quantize_nchw_kernel, but the input tile
// (8 rows of a x GBT*8 rows of b x HWT positions) arrives by one tiled TMA
// copy into a QT_STAGES-deep shared ring, filled by a producer warp while the
// eight compute warps quantize the previous tiles from shared memory.  The
// global-load latency then no longer waits on the encode work.
constexpr int QT_STAGES = 2;
constexpr int QT_CWARPS = 8;
constexpr int QT_THREADS = (QT_CWARPS + 1) * 32;

struct QtCtl {
  uint64_t full[QT_STAGES], empty[QT_STAGES];
  int coord[QT_STAGES][4];   // tile of each stage: position tile, b-group tile, a-group (set by the producer)
  int abort;
};

// bounded wait: gives up after 2 s, or at once when another warp has given
// up, so that every warp leaves its loop and the CTA still meets at its
// barriers
template <class Ctl>
__device__ __forceinline__ bool qt_wait(uint64_t *bar, uint32_t parity, Ctl *ctl, uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
    if (globaltimer_ns() - t0 > 2000000000ull) {
      atomicOr(status, ST_TIMEOUT);
      *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
      return false;
    }
  }
}

// The quantizing warps' loop over the CTA's tiles (see quantize_tma_kernel);
// returns the largest |x| seen (fp32 bits).  Each thread encodes one block
// and writes its payload and scale straight to global memory (16-byte
// stores; the eight warps of a tile write neighbouring blocks, so lines fill
// in L2 before they are written back), so the warps never wait on one
// another.  TINY: T_scale below 2^-62.
template <int FMT, typename T, int GBT, bool TINY>
__device__ __forceinline__ uint32_t tma_compute(const QuantParams &p, QtCtl *ctl, uint8_t *ring, int ntiles,
                                                int hw_tiles, int gb_tiles, float s_t) {
  constexpr int HWT = QN_HW * (QN_GB / GBT);
  constexpr int BB = Fmt<FMT>::BLOCK_BYTES;
  constexpr int STAGE = HWT * GBT * 64 * (int)sizeof(T);
  const int GA = (int)(p.d0 / 8), GB = (int)(p.d1 / 8);
  const int64_t HW = p.d2 * p.d3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wl = warp % GBT, hl = (warp / GBT) * 32 + lane;
  const float inv_den = block_den_rcp<FMT, TINY>(s_t);
  uint32_t my_amax = 0;
  int it = 0;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const int s = it % QT_STAGES;
    if (!qt_wait(&ctl->full[s], (it / QT_STAGES) & 1, ctl, p.status)) break;
    // the stage's tile, written by the producer before the copy's arrival
    // (read before this warp releases the stage)
    const int hwt = ctl->coord[s][0], gbt = ctl->coord[s][1], ga = ctl->coord[s][2];
    const int64_t hw0 = (int64_t)hwt * HWT;
    const int gb0 = gbt * GBT;
    const int ngb = min(GBT, GB - gb0);
    const int nhw = (int)(HW - hw0 < (int64_t)HWT ? HW - hw0 : (int64_t)HWT);
    // tile in shared memory: [a (8)][b (GBT*8)][hw (HWT)], hw fastest
    const T *tile = reinterpret_cast<const T *>(ring + s * STAGE) + (wl * 8) * HWT + hl;
    const bool mine = wl < ngb && hl < nhw;
    uint32_t raw[sizeof(T) == 2 ? 32 : 64];
    if (mine) {
#pragma unroll
      for (int a = 0; a < 8; ++a) {
#pragma unroll
        for (int b = 0; b < 8; b += (sizeof(T) == 2 ? 2 : 1)) {
          const T *q = tile + (a * GBT * 8 + b) * HWT;
          if (sizeof(T) == 2) {
            const uint32_t lo = *reinterpret_cast<const unsigned short *>(q);
            const uint32_t hi = *reinterpret_cast<const unsigned short *>(q + HWT);
            raw[(a * 8 + b) / 2] = lo | (hi << 16);
          } else {
            raw[a * 8 + b] = *reinterpret_cast<const uint32_t *>(q);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[s]);          // tile consumed (values are in registers)
    if (mine) {
      uint32_t mb = 0;
      if (sizeof(T) == 2) {
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) m2 = __vmaxu2(m2, raw[i] & 0x7FFF7FFFu);
        mb = max(m2 << 16, m2 & 0xFFFF0000u);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) mb = max(mb, raw[i & 63] & 0x7FFFFFFFu);
      }
      my_amax = max(my_amax, mb);
      if (mb >= 0x7F800000u) atomicOr(p.status, ST_NONFINITE);
      const int64_t blk = ((hw0 + hl) * GA + ga) * (int64_t)GB + gb0 + wl;
      RegRows<FMT> rows;
      const uint32_t bs_code = encode_raw_block<FMT, T, TINY>(raw, mb, s_t, inv_den, rows);
      rows.store(p.codes + blk * BB);
      p.scales[blk] = (uint8_t)bs_code;
    }
  }
  return my_amax;
}

// the tiny-T_scale loop, kept out of line (rare; inlined beside the common
// loop it would raise the register pressure of every launch)
template <int FMT, typename T, int GBT>
__device__ __noinline__ uint32_t tma_compute_tiny(const QuantParams &p, QtCtl *ctl, uint8_t *ring, int ntiles,
                                                  int hw_tiles, int gb_tiles, float s_t) {
  return tma_compute<FMT, T, GBT, true>(p, ctl, ring, ntiles, hw_tiles, gb_tiles, s_t);
}

template <int FMT, typename T, int GBT>
__global__ void __launch_bounds__(QT_THREADS, 2)
    quantize_tma_kernel(const __grid_constant__ CUtensorMap tm, QuantParams p, int ntiles, int hw_tiles, int gb_tiles) {
  constexpr int HWT = QN_HW * (QN_GB / GBT);
  constexpr int STAGE = HWT * GBT * 64 * (int)sizeof(T);
  extern __shared__ __align__(128) uint8_t qraw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(qraw) + 127) & ~uintptr_t(127));
  QtCtl *ctl = reinterpret_cast<QtCtl *>(ring + QT_STAGES * STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const float amax_src = __uint_as_float(*p.amax_src_bits);
  const float s_t = __fdiv_rn(amax_src, Fmt<FMT>::DENOM);
  if (threadIdx.x == 0) {
    for (int s = 0; s < QT_STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], QT_CWARPS);
    }
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (blockIdx.x == 0) {
      *p.s_t_out = s_t;
      if (!(amax_src <= 3.4028234663852886e38f)) atomicOr(p.status, ST_NONFINITE);
    }
  }
  __syncthreads();

  if (warp == QT_CWARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = it % QT_STAGES;
        if (!qt_wait(&ctl->empty[s], ((it / QT_STAGES) & 1) ^ 1, ctl, p.status)) break;
        // last tile first: after the exact-statistic pass, which reads the
        // tensor front to back, its tail is the part still in L2
        const int tr = ntiles - 1 - t;
        const int hwt = tr % hw_tiles, rest = tr / hw_tiles, gbt = rest % gb_tiles, ga = rest / gb_tiles;
        // the quantizing warps read the tile from here, not by dividing
        // themselves; the arrival below releases these writes
        ctl->coord[s][0] = hwt;
        ctl->coord[s][1] = gbt;
        ctl->coord[s][2] = ga;
        mbar_expect_tx(&ctl->full[s], STAGE);
        tma_load_3d(ring + s * STAGE, &tm, &ctl->full[s], hwt * HWT, gbt * GBT * 8, ga * 8);
      }
      for (int i = 0; i < QT_STAGES && i < it; ++i) {   // copies in flight land before exit
        const int q = it - 1 - i;
        mbar_wait(&ctl->full[q % QT_STAGES], (q / QT_STAGES) & 1, p.status);   // ignores the abort flag
      }
    }
    __syncwarp();
    return;
  }

  // --------------------------------------------------------------- compute
  const uint32_t my_amax =
      is_tiny_scale(s_t) ? tma_compute_tiny<FMT, T, GBT>(p, ctl, ring, ntiles, hw_tiles, gb_tiles, s_t)
                         : tma_compute<FMT, T, GBT, false>(p, ctl, ring, ntiles, hw_tiles, gb_tiles, s_t);
  if (p.amax_meas_bits) {
    uint32_t m = my_amax;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0 && m) atomicMax(p.amax_meas_bits, m);
  }
}

template <int FMT, typename T, int GBT>
static cudaError_t launch_tma_q(const T *src, const QuantParams &p, int num_sms, cudaStream_t s) {
  constexpr int HWT = QN_HW * (QN_GB / GBT);
  const int64_t HW = p.d2 * p.d3, GB = p.d1 / 8, GA = p.d0 / 8;
  alignas(64) uint8_t map[128];
  const uint64_t dims[3] = {(uint64_t)HW, (uint64_t)p.d1, (uint64_t)p.d0};
  const uint32_t box[3] = {(uint32_t)HWT, (uint32_t)(GBT * 8), 8u};
  if (!make_tensor_map(map, src, (int)sizeof(T), 3, dims, box)) return cudaErrorInvalidValue;
  const int64_t hw_tiles = (HW + HWT - 1) / HWT, gb_tiles = (GB + GBT - 1) / GBT;
  const int64_t ntiles = GA * gb_tiles * hw_tiles;
  constexpr size_t STAGE = (size_t)HWT * GBT * 64 * sizeof(T);
  const size_t smem = 128 + QT_STAGES * STAGE + sizeof(QtCtl);
  auto k = quantize_tma_kernel<FMT, T, GBT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, QT_THREADS, smem);
  const int64_t grid = std::min<int64_t>(ntiles, (int64_t)num_sms * std::max(1, per_sm));
  k<<<(unsigned)grid, QT_THREADS, smem, s>>>(*reinterpret_cast<const CUtensorMap *>(map), p, (int)ntiles,
                                             (int)hw_tiles, (int)gb_tiles);
  return cudaGetLastError();
}

// TMA path when the rows are 16-byte aligned and the ring fits, else the
// direct-load kernel
template <int FMT, typename T>
static bool try_tma_q(const T *src, const QuantParams &p, int num_sms, cudaStream_t s, cudaError_t &err) {
  const int64_t HW = p.d2 * p.d3, GB = p.d1 / 8;
  if ((HW * (int64_t)sizeof(T)) % 16 || (reinterpret_cast<uintptr_t>(src) & 15) || HW >= ((int64_t)1 << 31) ||
      p.d0 * p.d1 >= ((int64_t)1 << 31))
    return false;
  if (sizeof(T) == 4 && GB >= 8) return false;   // two 64 KB stages per CTA leave one CTA per SM; direct kernel
  if (GB >= 8) err = launch_tma_q<FMT, T, 8>(src, p, num_sms, s);
  else if (GB >= 4) err = launch_tma_q<FMT, T, 4>(src, p, num_sms, s);
  else if (GB >= 2) err = launch_tma_q<FMT, T, 2>(src, p, num_sms, s);
  else err = launch_tma_q<FMT, T, 1>(src, p, num_sms, s);
  return true;
}

// ----------------------------------------------------------------- launch
template <int FMT, typename T>
static cudaError_t launch_q(const void *src, int layout, const QuantParams &p, int num_sms, cudaStream_t s) {
  const int64_t nblk = (p.d0 / 8) * (p.d1 / 8) * p.d2 * p.d3;
  const T *x = static_cast<const T *>(src);
  if (layout == 1) {
    const unsigned grid = (unsigned)((nblk + 255) / 256);
    if (p.sr) quantize_kernel<FMT, T, 1, true><<<grid, 256, 0, s>>>(x, p);
    else quantize_kernel<FMT, T, 1, false><<<grid, 256, 0, s>>>(x, p);
    return cudaGetLastError();
  }
  cudaError_t err = cudaSuccess;
  if (!p.sr && try_tma_q<FMT, T>(x, p, num_sms, s, err)) return err;   // stochastic codes: direct-load kernel
  // NCHW / OIHW: GBT b-groups x 256 / GBT positions per CTA, contiguous output runs
  const int64_t HW = p.d2 * p.d3, GB = p.d1 / 8;
  const int64_t GBT = GB < QN_GB ? GB : QN_GB, HWT = QN_HW * (QN_GB / GBT);
  const int64_t grid = (p.d0 / 8) * ((GB + GBT - 1) / GBT) * ((HW + HWT - 1) / HWT);
  if (p.sr) quantize_nchw_kernel<FMT, T, true><<<(unsigned)grid, 256, 0, s>>>(x, p);
  else quantize_nchw_kernel<FMT, T, false><<<(unsigned)grid, 256, 0, s>>>(x, p);
  return cudaGetLastError();
}

// The decoded weight copy: row r of block b (eight codes) becomes the 16 bytes
// out[8 b + r], eight fp16 values code * B_scale (x 1/4 for E4M3 codes) --
// the conversion the convolutions' decode warps apply on chip (decode_raw,
// scale_pair), so a convolution that copies these rows computes exactly what
// it computes from the packed blocks.  One thread per row.
template <int F>
__global__ void __launch_bounds__(256) weight_decode_kernel(const uint8_t *__restrict__ codes,
                                                            const uint8_t *__restrict__ scales, int64_t rows,
                                                            uint4 *__restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < rows; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i >> 3;
    out[i] = decode_raw<F>(row8_bits<F>(codes + b * Fmt<F>::BLOCK_BYTES, (int)(i & 7)), scale_pair<F>(scales[b]));
  }
}

cudaError_t launch_weight_decode(const uint8_t *codes, const uint8_t *scales, int fmt, int64_t nblocks, void *out,
                                 int num_sms, cudaStream_t s) {
  const int64_t rows = nblocks * 8;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((rows + 255) / 256, (int64_t)num_sms * 8));
  uint4 *o = static_cast<uint4 *>(out);
  if (fmt == 4) weight_decode_kernel<4><<<grid, 256, 0, s>>>(codes, scales, rows, o);
  else if (fmt == 6) weight_decode_kernel<6><<<grid, 256, 0, s>>>(codes, scales, rows, o);
  else weight_decode_kernel<8><<<grid, 256, 0, s>>>(codes, scales, rows, o);
  return cudaGetLastError();
}

cudaError_t launch_amax(const void *src, int dtype, int64_t n, uint32_t *amax_bits, int num_sms, cudaStream_t s) {
  const int64_t per = dtype == 0 ? 4 : 8;
  int64_t want = (n / per + 255) / 256;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 8));
  if (dtype == 0) amax_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(src), n, amax_bits);
  else amax_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), n, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void *src, int dtype, int layout, int fmt, const QuantParams &p, int num_sms,
                            cudaStream_t s) {
  if (dtype == 0) {
    if (fmt == 4) return launch_q<4, float>(src, layout, p, num_sms, s);
    if (fmt == 6) return launch_q<6, float>(src, layout, p, num_sms, s);
    return launch_q<8, float>(src, layout, p, num_sms, s);
  }
  if (fmt == 4) return launch_q<4, __nv_bfloat16>(src, layout, p, num_sms, s);
  if (fmt == 6) return launch_q<6, __nv_bfloat16>(src, layout, p, num_sms, s);
  return launch_q<8, __nv_bfloat16>(src, layout, p, num_sms, s);
}

}  // namespace mq
