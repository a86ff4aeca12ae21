#pragma once
// conv_halo.cuh -- forward and data-gradient convolutions (stride 1 and 2)
// that decode every packed input block once per tile and reuse it for all
// taps: the kernel templates, instantiated by conv_halo_fwd.cu and
// conv_halo_dgrad.cu (in parallel translation units), and the wait helpers
// the weight-gradient kernel in conv_halo.cu shares.
//
// MicroQonv §IV-A builds the channel-batch-first im2col X' on chip: each
// contiguous CBF block crosses the off-chip/on-chip boundary once and is then
// replicated locally for every receptive field that needs it.  Here the
// replication costs nothing: a CTA
// tile covers R output rows x P output positions x G batch groups (8 n each)
// = R x 128 GEMM rows, and per chunk of 16 input channels the CTA stages the
// (R + Kh - 1) x (P + Kw - 1) halo of packed input blocks (TMA, zero fill
// outside the image), decodes it once to fp16 core matrices, and every tap
// (u, v) of every output row s reads the same decoded halo through a
// shared-memory matrix descriptor whose start address is shifted by
// ((s + u) * (P + Kw - 1) + v) halo positions.  The weights of the chunk
// (all taps, BN output channels) are staged and decoded the same way.
//
// Stride 2: the halo spans 2 (R - 1) + Kh rows and its even and odd input
// columns are staged as two phases (two TMA boxes through a [H][W/2][2]
// view of the codes), so output position p, tap v reads phase v % 2 at
// position p + v / 2: the rows of one tap are again unit-stride halo
// positions and one descriptor per tap still covers the 128 GEMM rows.
//
// The data gradient of a stride-1 layer is the same correlation run on dY
// with the taps mirrored and the weight blocks read transposed
// (MN-major descriptor), padding Kh - 1 - pad: dX = col2im(W^T G_Y) of
// MicroQonv §IV-A without any col2im buffer.  At stride 2 a tile covers
// output quads (2 x 2 dX pixels): dX[2i + a] sums W[kh] dY[i + (a + pad -
// kh) / 2] over the taps kh of parity a + pad, so each output phase (a, b)
// is a stride-1 correlation over dY with its own taps; the tile keeps one
// accumulator per (row, phase) and feeds each decoded tap to its phase.
//
// GEMM per tile: rows = (output row s, position p, batch group j, n), columns
// = output channels (BN), K = (chunk, tap, 16 channels).  One accumulator of
// 128 x BN fp32 per output row s lives in TMEM, in a ring of NS slots that
// fills the TMEM: row s of the k-th tile uses slot (k R + s) % NS, so while
// the epilogue drains one tile the next tile's rows already accumulate in
// the spare slots and in the slots drained first.
//
// Warp roles (conv kernel): warps 0-7 decode, warps 8-15 drain the
// accumulators (tcgen05.ld; warps w and w+4 share TMEM lane quadrant w % 4
// and take alternate 16- or 32-column chunks) into fp32 HWCN outputs or
// requantized CBF blocks, warp 16 copies block scales and issues the TMA
// loads (lane 0), lane 0 of warps 17 and 18 issue tcgen05.mma (the two
// issuers split a tile's accumulators: the issue loop of one thread, not
// the tensor pipe, bounds the MMA rate of a single issuer here).  The
// weight-gradient kernel has ten decode warps and one issuer.  Every wait is
// bounded; on expiry the CTA records MQ_ERR_TIMEOUT, stops, lets its copies
// and MMAs in flight finish and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <numeric>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mq {

namespace {

constexpr int HC_DEC_WARPS = 8;
constexpr int HC_EPI_WARP0 = 8;
constexpr int HC_EPI_WARPS = 8;   // two per TMEM lane quadrant, alternating 16-column chunks
constexpr int HC_TMA_WARP = 16;
constexpr int HC_MMA_WARP = 17;
// the conv kernel has a second MMA-issuing warp: output rows are split
// between the two issuers, so their issue loops run side by side
constexpr int HC_MMA_WARP2 = 18;
constexpr int HC_CONV_THREADS = 19 * 32;
constexpr int HC_DEC_THREADS = HC_DEC_WARPS * 32;
constexpr int CGC = 2;          // channel groups (8 channels each) per chunk: K = 16 per tap
constexpr int DSTAGES = 2;      // decoded ring depth
constexpr int MAX_PS = 4;       // packed ring depth (at most)
constexpr int MAX_R = 8;

struct HcCtl {
  uint64_t pfull[MAX_PS], pempty[MAX_PS];
  uint64_t dfull[DSTAGES], dempty[DSTAGES];
  uint64_t wfull[DSTAGES];   // decoded weight copy landed in the decoded stage (wd only)
  uint64_t sfull[2], sempty[2];
  uint64_t acc_full[MAX_R], acc_empty[MAX_R];
  uint64_t done;
  uint32_t tmem_base;
  volatile int abort_flag;
};

// Bounded wait for the phase of `bar` with the given parity: gives up after
// 2 s (records MQ_ERR_TIMEOUT and raises the CTA's abort flag), or at once
// when another warp of the CTA has given up.
__device__ __forceinline__ bool hc_wait(uint64_t *bar, uint32_t parity, const HaloConv &p, HcCtl *ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if ((it & 7u) == 7u) {
      if (ctl->abort_flag) return false;
      if (globaltimer_ns() - t0 > 2000000000ull) {
        atomicOr(p.status, ST_TIMEOUT);
        ctl->abort_flag = 1;
        return false;
      }
    }
  }
}

// Wait, within the same limit but whatever the abort flag says, for copies
// or MMAs this thread already issued: they land regardless, and must have
// landed before the CTA frees its TMEM or exits.
__device__ __forceinline__ bool hc_drain(uint64_t *bar, uint32_t parity, uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if ((it & 7u) == 7u && globaltimer_ns() - t0 > 2000000000ull) {
      atomicOr(status, ST_TIMEOUT);
      return false;
    }
  }
}

struct TileCoord {
  int g0, w0, h0, n0;   // first batch group, output column, output row, output channel
};

__device__ __forceinline__ TileCoord hc_tile(const HaloConv &p, int t) {
  TileCoord c;
  int r = t;
  c.g0 = (r % p.tiles_g) * p.G;
  r /= p.tiles_g;
  c.w0 = (r % p.tiles_w) * p.P;
  r /= p.tiles_w;
  c.h0 = (r % p.tiles_h) * p.R;
  r /= p.tiles_h;
  c.n0 = r * p.BN;
  return c;
}

// Requantize 8 NBK fp32 columns of one row into NBK blocks of the next
// layer's activations (see quantize.cu for the rounding).  Lanes 8q..8q+7
// hold the eight batch rows of one block; the block amax is their
// shuffle-max.  The per-block scale work (E4M3 block scale, bracket
// multipliers) is done once per block: lane 8q + j computes it for block
// j % NBK and the group reads it back by shuffles.  The blocks are processed
// side by side (independent chains).  TINY: T_scale below 2^-62, encoded from
// y 2^64 and T_scale 2^64 (s_t and inv_den are then the scaled ones; see up64).
template <int F, int NBK, bool TINY>
__device__ __forceinline__ void hc_requant(const HaloConv &p, const float *y, int64_t blk_pos_ng, int n_in, int co0,
                                           bool row_ok, float s_t, float inv_den, uint32_t &amax_acc) {
  static_assert(NBK == 2 || NBK == 4, "blocks side by side per chunk");
  // block amax of this lane's row: the fp32 max of |y|, a NaN (only from an
  // overflowed scale product) propagating, so that its bit pattern orders
  // above every finite value and Inf as the |y| bit patterns do
  float m[NBK];
#pragma unroll
  for (int h = 0; h < NBK; ++h) {
    float mm = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) mm = fmax_nan(mm, fabsf(y[8 * h + j]));
    m[h] = (row_ok && co0 + 8 * h < p.NC) ? mm : 0.0f;
  }
  // reduce-scatter over the 8 lanes (8 rows) of each block: lane j ends with
  // the amax of block j mod NBK, the block whose scale it computes
  const int lj = threadIdx.x & 7;
  float k;
  if constexpr (NBK == 4) {
    const bool b0 = lj & 1, b1 = lj & 2;
    float a = b0 ? m[1] : m[0], c = b0 ? m[3] : m[2];
    const float a_out = b0 ? m[0] : m[1], c_out = b0 ? m[2] : m[3];
    a = fmax_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a_out, 1));
    c = fmax_nan(c, __shfl_xor_sync(0xFFFFFFFFu, c_out, 1));
    k = b1 ? c : a;
    k = fmax_nan(k, __shfl_xor_sync(0xFFFFFFFFu, b1 ? a : c, 2));
  } else {
    const bool b0 = lj & 1;
    k = fmax_nan(b0 ? m[1] : m[0], __shfl_xor_sync(0xFFFFFFFFu, b0 ? m[0] : m[1], 1));
    k = fmax_nan(k, __shfl_xor_sync(0xFFFFFFFFu, k, 2));
  }
  k = fmax_nan(k, __shfl_xor_sync(0xFFFFFFFFu, k, 4));
  const uint32_t mine = __float_as_uint(k);
  amax_acc = max(amax_acc, mine);
  const float amax_mine = TINY ? up64(__uint_as_float(mine)) : __uint_as_float(mine);
  const uint32_t bsc_mine = block_scale_code_r<F>(amax_mine, s_t, inv_den);
  float lo_mine, hi_mine;
  quot_bracket(code_value<8>(bsc_mine), s_t, lo_mine, hi_mine);
  const int src0 = (threadIdx.x & 31) & ~7;
#pragma unroll
  for (int h = 0; h < NBK; ++h) {
    const int co = co0 + 8 * h;
    const uint32_t bsc = __shfl_sync(0xFFFFFFFFu, bsc_mine, src0 + h);
    const float inv_lo = __shfl_sync(0xFFFFFFFFu, lo_mine, src0 + h);
    const float inv_hi = __shfl_sync(0xFFFFFFFFu, hi_mine, src0 + h);
    const float bs = code_value<8>(bsc);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = TINY ? up64(y[8 * h + j]) : y[8 * h + j];
    const uint64_t bits = encode_row8_b<F>(v, bs, s_t, inv_lo, inv_hi);
    if (row_ok && co < p.NC) {
      const int64_t blk = blk_pos_ng + co / 8;
      store_row8<F>(p.rq.codes + blk * Fmt<F>::BLOCK_BYTES, n_in, bits);
      if (n_in == 0) p.rq.scales[blk] = (uint8_t)bsc;
    }
  }
}

// hc_requant with stochastically rounded element codes (MicroQonv §III-A; see
// encode_row8_sr): the block scales are decided exactly as in hc_requant
// (st_q, inv_den and `tiny` as there), the codes from q = fl32(|y| /
// fl32(B_scale s_t)) with the unscaled T_scale s_t and Philox key p.rq.sr_seed.
template <int F, int NBK>
__device__ __forceinline__ void hc_requant_sr(const HaloConv &p, const float *y, int64_t blk_pos_ng, int n_in, int co0,
                                              bool row_ok, float s_t, float st_q, float inv_den, bool tiny,
                                              uint32_t &amax_acc) {
  uint32_t m[NBK];
#pragma unroll
  for (int h = 0; h < NBK; ++h) {
    uint32_t mm = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mm = max(mm, __float_as_uint(y[8 * h + j]) & 0x7FFFFFFFu);
    m[h] = (row_ok && co0 + 8 * h < p.NC) ? mm : 0u;
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1)
#pragma unroll
    for (int h = 0; h < NBK; ++h) m[h] = max(m[h], __shfl_xor_sync(0xFFFFFFFFu, m[h], o));
  const int hb = n_in & (NBK - 1);
  uint32_t mine = m[0];
#pragma unroll
  for (int h = 1; h < NBK; ++h) mine = hb == h ? m[h] : mine;
  const float amax_mine = tiny ? up64(__uint_as_float(mine)) : __uint_as_float(mine);
  const uint32_t bsc_mine = block_scale_code_r<F>(amax_mine, st_q, inv_den);
  const int src0 = (threadIdx.x & 31) & ~7;
#pragma unroll
  for (int h = 0; h < NBK; ++h) {
    amax_acc = max(amax_acc, m[h]);
    const int co = co0 + 8 * h;
    const uint32_t bsc = __shfl_sync(0xFFFFFFFFu, bsc_mine, src0 + h);
    const float d = __fmul_rn(code_value<8>(bsc), s_t);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = y[8 * h + j];
    if (row_ok && co < p.NC) {
      const int64_t blk = blk_pos_ng + co / 8;
      store_row8<F>(p.rq.codes + blk * Fmt<F>::BLOCK_BYTES, n_in, encode_row8_sr<F>(v, d, p.rq.sr_seed, blk, n_in));
      if (n_in == 0) p.rq.scales[blk] = (uint8_t)bsc;
    }
  }
}

// One accumulator row chunk of W columns (W = 16 or 32) starting at column
// c0: scaled fp32 HWCN stores and / or the fused requantization.  RARE: the
// stochastic and tiny-T_scale requantizations are compiled in (only in the
// out-of-line epilogue copy that launches needing them run).
template <int FR, int W, bool RARE>
__device__ __forceinline__ void hc_epi_chunk(const HaloConv &p, uint32_t taddr, bool zero, float f, int64_t obase,
                                             int64_t rq_blk, int n_in, int co0, bool valid, float rq_st,
                                             float rq_inv, bool rq_tiny, float rq_st_true, uint32_t &amax_acc) {
  float y[W];
  if (zero) {   // accumulator never written (warp-uniform)
#pragma unroll
    for (int jj = 0; jj < W; ++jj) y[jj] = 0.0f;
  } else {
    uint32_t r[W];
    if constexpr (W == 32) tmem_ld32(taddr, r);
    else tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int jj = 0; jj < W; jj += 2) mul2(__uint_as_float(r[jj]), __uint_as_float(r[jj + 1]), f, y[jj], y[jj + 1]);
  }
  if (p.out && valid) {
    float *o = p.out + obase + (int64_t)co0 * p.N;
#pragma unroll
    for (int jj = 0; jj < W; ++jj)
      if (co0 + jj < p.NC) o[(int64_t)jj * p.N] = y[jj];
  }
  if constexpr (FR != 0) {
    if constexpr (RARE) {
      if (p.rq.sr)
        hc_requant_sr<FR, W / 8>(p, y, rq_blk, n_in, co0, valid, rq_st_true, rq_st, rq_inv, rq_tiny, amax_acc);
      else if (rq_tiny) hc_requant<FR, W / 8, true>(p, y, rq_blk, n_in, co0, valid, rq_st, rq_inv, amax_acc);
      else hc_requant<FR, W / 8, false>(p, y, rq_blk, n_in, co0, valid, rq_st, rq_inv, amax_acc);
    } else {
      hc_requant<FR, W / 8, false>(p, y, rq_blk, n_in, co0, valid, rq_st, rq_inv, amax_acc);
    }
  }
}

}  // namespace

// MMA issuers (see the kernel); QDM: the stride-2 data gradient in output quads
template <int OP, bool QDM>
__device__ __forceinline__ void hc_issue(const HaloConv &p, HcCtl *ctl, uint8_t *smem, uint32_t tmem, int warp, int lane) {
  // ---------------------------------------------------------- MMA issuers
  // issuer i (lane 0 of warp HC_MMA_WARP + i) takes the accumulators
  // i, i + NI, ... of a tile (output rows; with QD, (row, phase) pairs);
  // both wait for each decoded stage and each commits its MMAs to the
  // stage's release barrier (count NI)
  const int issuer = warp - HC_MMA_WARP, NI = p.RT >= 2 ? 2 : 1;
  if (lane == 0 && issuer < NI) {
    const uint32_t idesc = idesc_f16(128, p.BN, false, OP == OP_DGRAD);
    // Descriptor words: the high word (stride fields, version) is fixed;
    // the low word holds (address >> 4) in bits 0-13, so moving an operand
    // by `bytes` adds bytes >> 4 to it (addresses stay below 256 KB).
    const uint64_t a_desc = sdesc(smem_u32(smem + p.off_dec), 128, CGC * 128);
    const uint64_t b_desc = OP == OP_FWD ? sdesc(smem_u32(smem + p.off_dec + p.dec_b_off), 128, CGC * 128)
                                         : sdesc(smem_u32(smem + p.off_dec + p.dec_b_off), p.NB * 128, 128);
    const uint32_t a_hi = (uint32_t)(a_desc >> 32), b_hi = (uint32_t)(b_desc >> 32);
    const uint32_t d_row = (uint32_t)((p.WP * p.G * CGC * 128) >> 4);     // one halo row
    const uint32_t d_col = (uint32_t)((p.G * CGC * 128) >> 4);            // one halo position
    const uint32_t d_phase = (uint32_t)((p.PHP * p.G * CGC * 128) >> 4);  // one column phase
    const uint32_t d_tap = (uint32_t)((p.NB * CGC * 128) >> 4);           // one weight tap
    const uint32_t d_stage = p.dec_stage >> 4;
    const int sh = p.S - 1;   // tap v sits in column phase v & sh, v >> sh positions in
    const int taps = p.Kh * p.Kw;
    // Per-tap operand offsets, built once: tap t = (u, v) reads the halo
    // at row u, phase v & sh, position v >> sh, and the weights of tap t
    // (fwd) or of the mirrored tap taps - 1 - t (dgrad).  Up to UT taps
    // the issue loop is unrolled over this table: one add per operand per
    // MMA.
    // With QD the table is in phase order: entry j is tap qorder[j], whose
    // dY offsets (dh, dw) = ((a + pad - kh) / 2, (b + pad - kw) / 2) are
    // taken from the halo origin (-padh, -padw).
    constexpr int UT = 9;
    uint32_t a_off[UT], b_off[UT];
#pragma unroll
    for (int t = 0; t < UT; ++t) {
      if (QDM) {
        const int tq = p.qorder[t], u = tq / p.Kw, v = tq - u * p.Kw;
        const int ah = ((u - p.qpad) % 2 + 2) % 2, aw = ((v - p.qpad) % 2 + 2) % 2;
        const int dh = (ah + p.qpad - u) / 2 + p.padh, dw = (aw + p.qpad - v) / 2 + p.padw;
        a_off[t] = (uint32_t)dh * d_row + (uint32_t)dw * d_col;
        b_off[t] = (uint32_t)tq * d_tap;
      } else {
        const int u = t / p.Kw, v = t - u * p.Kw;
        a_off[t] = (uint32_t)u * d_row + (uint32_t)(v & sh) * d_phase + (uint32_t)(v >> sh) * d_col;
        b_off[t] = (uint32_t)(OP == OP_FWD ? t : taps - 1 - t) * d_tap;
      }
    }
    int dit = 0, k = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++k) {
      for (int c = 0; c < p.nchunks; ++c, ++dit) {
        const int ds = dit % DSTAGES;
        if (!hc_wait(&ctl->dfull[ds], (dit / DSTAGES) & 1, p, ctl)) { ok = false; break; }
        if (p.wd && !hc_wait(&ctl->wfull[ds], (dit / DSTAGES) & 1, p, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_stage = (uint32_t)a_desc + (uint32_t)ds * d_stage;
        const uint32_t b_stage = (uint32_t)b_desc + (uint32_t)ds * d_stage;
        // the weight descriptors of the chunk, shared by all its rows
        uint32_t bq[UT];
#pragma unroll
        for (int tp = 0; tp < UT; ++tp) bq[tp] = b_stage + b_off[tp];
        for (int sl = issuer; sl < p.RT && ok; sl += NI) {
          // accumulator ring: accumulator sl of the k-th tile uses slot
          // (k RT + sl) % NS; it is output row s = sl / NPHS (phase
          // f = gray(sl % 4) with QD)
          const int ring = k * p.RT + sl, slot = ring & (p.NS - 1), use = ring >> p.ns_log2;
          const int s = QDM ? sl >> 2 : sl;   // NPHS = 4 with QD, else 1
          if (c == 0) {
            if (!hc_wait(&ctl->acc_empty[slot], (use & 1) ^ 1, p, ctl)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t d = tmem + slot * p.acc_cols;
          const uint32_t a_s = a_stage + (uint32_t)(s * p.S) * d_row;
          if (QDM) {
            const int f = (sl & 3) ^ ((sl & 3) >> 1);
            const int beg = p.qbeg[f], end = p.qbeg[f + 1];
#pragma unroll
            for (int j = 0; j < UT; ++j)
              if (j >= beg && j < end)
                umma_f16(d, desc_of(a_hi, a_s + a_off[j]), desc_of(b_hi, bq[j]), idesc, (j > beg || c > 0) ? 1u : 0u);
          } else if (taps == UT) {   // 3x3: no per-tap predicate
            umma_f16(d, desc_of(a_hi, a_s + a_off[0]), desc_of(b_hi, bq[0]), idesc, c > 0 ? 1u : 0u);
#pragma unroll
            for (int tp = 1; tp < UT; ++tp) umma_f16_acc(d, desc_of(a_hi, a_s + a_off[tp]), desc_of(b_hi, bq[tp]), idesc);
          } else if (taps < UT) {
#pragma unroll
            for (int tp = 0; tp < UT; ++tp)
              if (tp < taps)
                umma_f16(d, desc_of(a_hi, a_s + a_off[tp]), desc_of(b_hi, bq[tp]), idesc, (tp > 0 || c > 0) ? 1u : 0u);
          } else {
            for (int tp = 0; tp < taps; ++tp) {
              const int u = tp / p.Kw, v = tp - u * p.Kw;
              const uint32_t ao = (uint32_t)u * d_row + (uint32_t)(v & sh) * d_phase + (uint32_t)(v >> sh) * d_col;
              const uint32_t bo = (uint32_t)(OP == OP_FWD ? tp : taps - 1 - tp) * d_tap;
              umma_f16(d, desc_of(a_hi, a_s + ao), desc_of(b_hi, b_stage + bo), idesc, (tp > 0 || c > 0) ? 1u : 0u);
            }
          }
          if (c == p.nchunks - 1) umma_commit(&ctl->acc_full[slot]);
        }
        umma_commit(&ctl->dempty[ds]);
      }
    }
    umma_commit(&ctl->done);
    hc_drain(&ctl->done, 0, p.status);   // every MMA issued so far has completed
  }
  __syncwarp();
}

// Epilogue warps (see the kernel); QDM: the stride-2 data gradient in output
// quads; RARE as in hc_epi_chunk
template <int FR, bool QDM, bool RARE>
__device__ __forceinline__ void hc_epilogue(const HaloConv &p, HcCtl *ctl, uint32_t tmem, int warp, int lane) {
  // ------------------------------------------------------------- epilogue
  const int q = warp & 3;                       // TMEM lanes 32q .. 32q+31
  const int half = (warp - HC_EPI_WARP0) >> 2;  // 16-column chunks half, half + 2, ...
  const int row = q * 32 + lane;
  const int g = row >> 3, n_in = row & 7, pp = g / p.G, j = g - pp * p.G;
  const float f = (*p.sa) * (*p.sb) * p.pre_mult;
  float rq_st = 0.0f;    // T_scale of the requantized output (stored unscaled)
  float rq_stq = 0.0f;   // the T_scale the quotients are formed with (x 2^64 when tiny)
  float rq_inv = 0.0f;
  bool rq_tiny = false;
  if (FR) {
    rq_st = __fdiv_rn(*p.rq.amax_in, Fmt<FR ? FR : 4>::DENOM);
    rq_tiny = is_tiny_scale(rq_st);
    rq_stq = rq_tiny ? rq_st * TINY_MULT : rq_st;
    rq_inv = __frcp_rn(Fmt<FR ? FR : 4>::EMAX * rq_stq);
  }
  uint32_t amax_acc = 0;
  int k = 0;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++k) {
    const TileCoord tc = hc_tile(p, t);
    const int ng = tc.g0 + j, n = ng * 8 + n_in;
    bool stop = false;
    for (int sl = 0; sl < p.RT; ++sl) {
      const int ring = k * p.RT + sl, slot = ring & (p.NS - 1), use = ring >> p.ns_log2;
      if (!hc_wait(&ctl->acc_full[slot], use & 1, p, ctl)) { stop = true; break; }
      tc_fence_after();
      int ho = tc.h0 + (QDM ? sl >> 2 : sl), wo = tc.w0 + pp;
      bool zero = false;
      if (QDM) {
        // output phase f = gray(sl % 4) = 2 a + b: dX pixel (2 ho + a, 2 wo + b);
        // a phase no tap reaches is zero
        const int fq = (sl & 3) ^ ((sl & 3) >> 1);
        ho = 2 * ho + (fq >> 1);
        wo = 2 * wo + (fq & 1);
        zero = p.qbeg[fq + 1] == p.qbeg[fq];
      }
      const bool valid = ho < p.outH && wo < p.outW;
      const int64_t pos = (int64_t)ho * p.outW + wo;
      const int64_t obase = pos * p.NC * (int64_t)p.N + n;
      const int64_t rq_blk = (pos * p.NG + ng) * p.NCG;
      const uint32_t tb = tmem + slot * p.acc_cols + ((uint32_t)(q * 32) << 16);
      // the two warps of a lane quadrant take alternate column chunks: 32
      // columns (four blocks side by side) for a requantize-only epilogue
      // when BN is a multiple of 64, else 16
      if (FR != 0 && !p.out && p.BN % 64 == 0) {
        for (int c0 = 32 * half; c0 < p.BN; c0 += 64)
          hc_epi_chunk<FR, 32, RARE>(p, tb + c0, zero, f, obase, rq_blk, n_in, tc.n0 + c0, valid, rq_stq, rq_inv,
                               rq_tiny, rq_st, amax_acc);
      } else {
        for (int c0 = 16 * half; c0 < p.BN; c0 += 32)
          hc_epi_chunk<FR, 16, RARE>(p, tb + c0, zero, f, obase, rq_blk, n_in, tc.n0 + c0, valid, rq_stq, rq_inv,
                               rq_tiny, rq_st, amax_acc);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty[slot]);
    }
    if (stop) break;
  }
  if (FR) {
#pragma unroll
    for (int o = 16; o; o >>= 1) amax_acc = max(amax_acc, __shfl_xor_sync(0xFFFFFFFFu, amax_acc, o));
    if (lane == 0 && amax_acc && p.rq.amax_out_bits) atomicMax(p.rq.amax_out_bits, amax_acc);
    if (blockIdx.x == 0 && row == 0 && half == 0) *p.rq.s_t_out = rq_st;
  }
}

// the epilogue copy with the stochastic and tiny-T_scale requantizations,
// kept out of line so that the common epilogue carries none of their code
template <int FR, bool QDM>
__device__ __noinline__ void hc_epilogue_rare(const HaloConv &p, HcCtl *ctl, uint32_t tmem, int warp, int lane) {
  hc_epilogue<FR, QDM, true>(p, ctl, tmem, warp, lane);
}

// the epilogue warps' entry: one launch-uniform choice of the epilogue copy
template <int FR, bool QDM>
__device__ __forceinline__ void hc_epilogue_entry(const HaloConv &p, HcCtl *ctl, uint32_t tmem, int warp, int lane) {
  if constexpr (FR != 0) {
    if (p.rq.sr || is_tiny_scale(__fdiv_rn(*p.rq.amax_in, Fmt<FR ? FR : 4>::DENOM))) {
      hc_epilogue_rare<FR, QDM>(p, ctl, tmem, warp, lane);
      return;
    }
  }
  hc_epilogue<FR, QDM, false>(p, ctl, tmem, warp, lane);
}


// FA: format of the input blocks (X or dY), FB: of the weights, FR: format of
// the fused requantization of the output (0 = none).
template <int OP, int FA, int FB, int FR>
__global__ void __launch_bounds__(HC_CONV_THREADS, 1)
    halo_conv_kernel(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_w,
                     const HaloConv p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  HcCtl *ctl = reinterpret_cast<HcCtl *>(smem + p.off_ctl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int BBA = Fmt<FA>::BLOCK_BYTES, BBB = Fmt<FB>::BLOCK_BYTES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.PS; ++s) {
      mbar_init(&ctl->pfull[s], 1);
      mbar_init(&ctl->pempty[s], HC_DEC_WARPS);
    }
    for (int s = 0; s < DSTAGES; ++s) {
      mbar_init(&ctl->dfull[s], HC_DEC_WARPS);
      mbar_init(&ctl->dempty[s], p.RT >= 2 ? 2 : 1);   // one commit per issuer
      mbar_init(&ctl->wfull[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->sfull[s], 64);
      mbar_init(&ctl->sempty[s], HC_DEC_WARPS);
    }
    // test support (INJECT_WITHHOLD_ACC_RELEASE): CTA 0's first accumulator
    // slot expects one release more than its epilogue warps give, so the
    // issuer's wait to reuse it can only expire; set here, the injection
    // costs the loops nothing
    const int extra = p.inject == INJECT_WITHHOLD_ACC_RELEASE && blockIdx.x == 0 ? 1 : 0;
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&ctl->acc_full[s], 1);
      mbar_init(&ctl->acc_empty[s], HC_EPI_WARPS + (s == 0 ? extra : 0));
    }
    mbar_init(&ctl->done, p.RT >= 2 ? 2 : 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == HC_MMA_WARP) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == HC_TMA_WARP) {
    // ------------------------------------------------------- TMA producer
    // Per tile the whole warp copies the halo block scales (zero outside the
    // image, where the TMA zero-fills the codes too) and the weight block
    // scales asynchronously into the tile's scale buffer (64 arrivals: two
    // per lane); lane 0 then streams the packed codes of every chunk, and
    // with the decoded weight copy lane 1 streams the chunks' weights.
    int pit = 0, wit = 0, k = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++k) {
      const TileCoord tc = hc_tile(p, t);
      const int tb = k & 1;
      int okw = 1;
      if (lane == 0) okw = hc_wait(&ctl->sempty[tb], ((k >> 1) & 1) ^ 1, p, ctl) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, okw, 0)) break;
      uint8_t *scd = smem + p.off_sc + tb * p.sc_stride;
      {
        // halo block scales: one run of G * CGin bytes per halo position,
        // positions ordered (column phase, row, column) like the code boxes;
        // the padding positions at the end of a phase get zeros
        const int run = p.G * p.CGin;
        copy_runs_rt(
            p.gran_h, scd, p.NPH * p.PHP, run, run,
            [&](int r) -> const uint8_t * {
              const int ph = r / p.PHP, rr = r - ph * p.PHP;
              const int hr = rr / p.WP, wc = rr - hr * p.WP;
              if (hr >= p.RH) return nullptr;
              const int hi = p.S * tc.h0 - p.padh + hr, wi = p.S * tc.w0 - p.padw + ph + p.S * wc;
              if ((unsigned)hi >= (unsigned)p.Hin || (unsigned)wi >= (unsigned)p.Win) return nullptr;
              return p.in_scales + (((int64_t)hi * p.Win + wi) * p.NG + tc.g0) * p.CGin;
            },
            [&](int) { return run; }, p.in_scales, lane);
        // weight block scales of the tile's output channels (none with the
        // decoded copy, which has them applied)
        const int nb0 = tc.n0 / 8;
        if (OP == OP_FWD && !p.wd) {
          const int nbv = min(p.NB, p.COG - nb0), fill = p.NB * p.CIG;
          copy_runs_rt(
              p.gran_w, scd + p.scw_off, p.Kh * p.Kw, fill, fill,
              [&](int tap) -> const uint8_t * { return p.w_scales + ((int64_t)tap * p.COG + nb0) * p.CIG; },
              [&](int) { return nbv * p.CIG; }, p.w_scales, lane);
        } else if (!p.wd) {
          const int nbv = min(p.NB, p.CIG - nb0);
          copy_runs_rt(
              p.gran_w, scd + p.scw_off, p.Kh * p.Kw * p.COG, p.NB, p.NB,
              [&](int r) -> const uint8_t * { return p.w_scales + (int64_t)r * p.CIG + nb0; },
              [&](int) { return nbv; }, p.w_scales, lane);
        }
        cp_async_arrive(&ctl->sfull[tb]);
        mbar_arrive(&ctl->sfull[tb]);
      }
      if (lane == 0) {
        for (int c = 0; c < p.nchunks; ++c, ++pit) {
          const int ps = pit % p.PS;
          if (!hc_wait(&ctl->pempty[ps], ((pit / p.PS) & 1) ^ 1, p, ctl)) { ok = false; break; }
          mbar_expect_tx(&ctl->pfull[ps], p.pk_bytes);
          uint8_t *dst = smem + p.off_pk + ps * p.pk_stage;
          if (p.S == 1) {
            tma_load_4d(dst, &tm_in, &ctl->pfull[ps], c * CGC * BBA / 8, tc.g0, tc.w0 - p.padw, tc.h0 - p.padh);
          } else {
            // stride 2: halo phase ph holds the input columns 2 w0 - padw + ph + 2 k,
            // read through the view [H][W/2][2][NG][..] of the same codes
            const uint32_t ph_bytes = (uint32_t)(p.PHP * p.G * CGC * BBA);   // a multiple of 128
            for (int ph = 0; ph < p.NPH; ++ph) {
              const int wc0 = 2 * tc.w0 - p.padw + ph, gph = wc0 & 1;
              tma_load_5d(dst + ph * ph_bytes, &tm_in, &ctl->pfull[ps], c * CGC * BBA / 8, tc.g0, gph,
                          (wc0 - gph) / 2, 2 * tc.h0 - p.padh);
            }
          }
          if (OP == OP_FWD && !p.wd)
            tma_load_3d(dst + p.pk_b_off, &tm_w, &ctl->pfull[ps], c * CGC * BBB / 8, tc.n0 / 8, 0);
          else if (!p.wd)
            tma_load_3d(dst + p.pk_b_off, &tm_w, &ctl->pfull[ps], (tc.n0 / 8) * BBB / 8, c * CGC, 0);
        }
      } else if (lane == 1 && p.wd) {
        // the decoded weight copy, straight into the weight half of each
        // decoded stage once the MMAs have released it (its own barrier, so
        // that it can be drained whatever the decode warps do)
        for (int c = 0; c < p.nchunks; ++c, ++wit) {
          const int ds = wit % DSTAGES;
          if (!hc_wait(&ctl->dempty[ds], ((wit / DSTAGES) & 1) ^ 1, p, ctl)) { ok = false; break; }
          mbar_expect_tx(&ctl->wfull[ds], p.wd_bytes);
          uint8_t *dst = smem + p.off_dec + ds * p.dec_stage + p.dec_b_off;
          if (OP == OP_FWD)
            tma_load_4d(dst, &tm_w, &ctl->wfull[ds], 0, c * CGC, tc.n0 / 8, 0);
          else
            tma_load_4d(dst, &tm_w, &ctl->wfull[ds], 0, tc.n0 / 8, c * CGC, 0);
        }
      }
      const int okv = ok ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, okv, 0) != 0 && __shfl_sync(0xFFFFFFFFu, okv, 1) != 0;
      pit = __shfl_sync(0xFFFFFFFFu, pit, 0);
      wit = __shfl_sync(0xFFFFFFFFu, wit, 1);
    }
    // let the copies in flight land before the CTA can exit: the last boxes
    // (whatever the abort flag says) and this warp's scale copies
    if (lane == 0) {
      for (int i = 0; i < p.PS && i < pit; ++i) {
        const int q = pit - 1 - i;
        hc_drain(&ctl->pfull[q % p.PS], (q / p.PS) & 1, p.status);
      }
    } else if (lane == 1) {
      for (int i = 0; i < DSTAGES && i < wit; ++i) {
        const int q = wit - 1 - i;
        hc_drain(&ctl->wfull[q % DSTAGES], (q / DSTAGES) & 1, p.status);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else if (warp < HC_DEC_WARPS) {
    // ------------------------------------------------------------ decoders
    const int tid = threadIdx.x;
    int pit = 0, dit = 0, k = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++k) {
      const TileCoord tc = hc_tile(p, t);
      const int tb = k & 1;
      if (!hc_wait(&ctl->sfull[tb], (k >> 1) & 1, p, ctl)) break;
      const uint8_t *sc = smem + p.off_sc + tb * p.sc_stride;
      for (int c = 0; c < p.nchunks; ++c, ++pit, ++dit) {
        const int ps = pit % p.PS, ds = dit % DSTAGES;
        if (!hc_wait(&ctl->pfull[ps], (pit / p.PS) & 1, p, ctl)) { ok = false; break; }
        if (!hc_wait(&ctl->dempty[ds], ((dit / DSTAGES) & 1) ^ 1, p, ctl)) { ok = false; break; }
        const uint8_t *pk = smem + p.off_pk + ps * p.pk_stage;
        uint8_t *dec = smem + p.off_dec + ds * p.dec_stage;
        // input halo: block (hr, wc, j, kc) at index ((hr * WP + wc) * G + j) * CGC + kc
        const int nh = p.nh_blocks * 8;
        // unrolled: two (halo) and four (weight) rows' shared loads in flight
        // per thread ahead of their conversions (measured: fwd 3%, dgrad 4%)
#pragma unroll 2
        for (int i = tid; i < nh; i += HC_DEC_THREADS) {
          const int blk = i >> 3, r = i & 7;
          const int hp = blk / CGC, kc = blk - hp * CGC;
          const uint8_t s = sc[hp * p.CGin + c * CGC + kc];
          const uint4 v = decode_raw<FA>(row8_bits<FA>(pk + blk * BBA, r), scale_pair<FA>(s));
          *reinterpret_cast<uint4 *>(dec + i * 16) = v;
        }
        // weights: fwd block (tap, nb, kc) at (tap * NB + nb) * CGC + kc;
        //          dgrad block (tap, kc, nb) at (tap * CGC + kc) * NB + nb
        const int nbr = p.wd ? 0 : p.nb_blocks * 8;   // the decoded copy arrives by TMA
        uint8_t *decb = dec + p.dec_b_off;
        const uint8_t *pkb = pk + p.pk_b_off;
        const uint8_t *scw = sc + p.scw_off;
        // dgrad: block (tap, kc, nb) has scale (tap * COG + c * CGC + kc) * NB + nb
        // = blk + tap * (COG - CGC) * NB + c * CGC * NB; tap = blk / (CGC * NB)
        // is carried along the thread's stride instead of divided out per row
        const int tap_span = CGC * p.NB, step_blk = HC_DEC_THREADS / 8;
        const int q_step = step_blk / tap_span, r_step = step_blk - q_step * tap_span;
        int d_tap = (tid >> 3) / tap_span, d_rem = (tid >> 3) - d_tap * tap_span;
#pragma unroll 4
        for (int i = tid; i < nbr; i += HC_DEC_THREADS) {
          const int blk = i >> 3, r = i & 7;
          int si;
          if (OP == OP_FWD) {   // block (tap, nb, kc); scales [tap][nb][cig]
            const int tn = blk / CGC, kc = blk - tn * CGC;
            si = tn * p.CIG + c * CGC + kc;
          } else {              // block (tap, kc, nb); scales [tap][cog][nb]
            si = blk + (d_tap * (p.COG - CGC) + c * CGC) * p.NB;
            // advance (d_tap, d_rem) by step_blk blocks without a loop, so the
            // row loop stays straight-line
            d_tap += q_step;
            d_rem += r_step;
            const bool wrap = d_rem >= tap_span;
            d_rem -= wrap ? tap_span : 0;
            d_tap += wrap ? 1 : 0;
          }
          const uint8_t s = scw[si];
          const uint4 v = decode_raw<FB>(row8_bits<FB>(pkb + blk * BBB, r), scale_pair<FB>(s));
          *reinterpret_cast<uint4 *>(decb + i * 16) = v;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl->pempty[ps]);
          mbar_arrive(&ctl->dfull[ds]);
        }
      }
      if (ok) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->sempty[tb]);
      }
    }
  } else if (warp == HC_MMA_WARP || warp == HC_MMA_WARP2) {
    if (OP == OP_DGRAD && p.QD) hc_issue<OP, true>(p, ctl, smem, tmem, warp, lane);
    else hc_issue<OP, false>(p, ctl, smem, tmem, warp, lane);
  } else if (warp >= HC_EPI_WARP0 && warp < HC_EPI_WARP0 + HC_EPI_WARPS) {
    if (OP == OP_DGRAD && p.QD) hc_epilogue_entry<FR, true>(p, ctl, tmem, warp, lane);
    else hc_epilogue_entry<FR, false>(p, ctl, tmem, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == HC_MMA_WARP) tmem_dealloc(tmem, 512);
}

// launch of one instantiation, and the dispatch over the operand formats
namespace {

template <int OP, int FA, int FB, int FR>
cudaError_t hc_launch(const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h, int grid,
                      cudaStream_t st) {
  auto k = halo_conv_kernel<OP, FA, FB, FR>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h.smem);
  if (e != cudaSuccess) return e;
  k<<<grid, HC_CONV_THREADS, h.smem, st>>>(a, b, h);
  return cudaGetLastError();
}

template <int OP, int FA, int FR>
cudaError_t hc_dispatch_b(int fb, const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h, int grid,
                          cudaStream_t st) {
  switch (fb) {
    case 4: return hc_launch<OP, FA, 4, FR>(a, b, h, grid, st);
    case 6: return hc_launch<OP, FA, 6, FR>(a, b, h, grid, st);
    default: return hc_launch<OP, FA, 8, FR>(a, b, h, grid, st);
  }
}

template <int OP, int FR>
cudaError_t hc_dispatch(int fa, int fb, const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h, int grid,
                        cudaStream_t st) {
  switch (fa) {
    case 4: return hc_dispatch_b<OP, 4, FR>(fb, a, b, h, grid, st);
    case 6: return hc_dispatch_b<OP, 6, FR>(fb, a, b, h, grid, st);
    default: return hc_dispatch_b<OP, 8, FR>(fb, a, b, h, grid, st);
  }
}

}  // namespace

}  // namespace mq
