// conv.cu -- implicit-im2col convolution GEMMs on packed channel-batch-first blocks.
//
// MicroQonv §IV-A writes the three GEMMs of a training step on the
// channel-batch-first layout as
//     Y_{Cout,N}     = W_{Cout,Cin}   . X'_{Cin,N}        (forward)
//     G_W{Cout,Cin}  = G_Y{Cout,N}    . X'^T_{Cin,N}      (weight gradient)
//     G_X'{Cin,N}    = W^T_{Cout,Cin} . G_Y{Cout,N}       (data gradient)
// with X' the im2col of X generated on chip from contiguous CBF blocks, and
// §IV-B aligns every reduction with an edge of the square 8x8 quantization
// block.  Here each 8x8 block is exactly one tcgen05 "core matrix" (8 rows x
// 16 bytes of fp16): a block decodes, row by row, to 64 fp16 values
// code * B_scale (exact), the tensor-core accumulates in fp32 in TMEM, and the
// epilogue multiplies by T_scale(A) * T_scale(B) -- the blockwise scaled dot
// product of MicroQonv §III-B, Eq. 7, with the block scales folded into the
// decoded operands.  Whether a block's fast axis is the reduction axis (K) or
// the row axis (M/N) is absorbed by the K-major / MN-major operand descriptor,
// so no block is ever transposed or quantized a second time.
//
// GEMM mapping (rows = TMEM lanes, columns = TMEM columns, K = reduction):
//   fwd   rows (out position, n)   cols c_out          K (tap, c_in)    A=X  K-major, B=W  K-major
//   dgrad rows (in position, n)    cols c_in           K (tap, c_out)   A=dY K-major, B=W  MN-major
//   wgrad rows c_out               cols (tap, c_in)    K (position, n)  A=dY MN-major, B=X MN-major
// dgrad walks the stride phases of the input so every tile only visits the
// taps that reach it; wgrad splits K and reduces partial sums in a fixed order.
//
// Warp roles of the persistent CTA: warps 0-7 decode packed blocks into a
// STAGES-deep shared-memory ring, warp 12 (one lane) issues tcgen05.mma into
// one of two TMEM accumulators, warps 8-11 drain the other accumulator
// (tcgen05.ld) and store fp32 results or requantize them.  Every mbarrier
// wait is bounded; on expiry the CTA records MQ_ERR_TIMEOUT and unwinds.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace mq {

constexpr int KCH = CONV_KCH;             // k-groups (8 reduction elements each) per stage: K = 64
constexpr int PROD_WARPS = 8;
constexpr int EPI_WARPS = 4;
constexpr int MMA_WARP = PROD_WARPS + EPI_WARPS;
constexpr int CONV_THREADS = (PROD_WARPS + EPI_WARPS + 1) * 32;
constexpr int STAGES = 4;
constexpr int A_STAGE = 16 * KCH * 128;   // 128 rows x 64 K x fp16

// packed row fetch from global memory (the decode itself is in common.cuh)
template <int F> __device__ __forceinline__ uint2 load_raw(const uint8_t *blk, int r) {
  if (F == 4) return make_uint2(__ldg(reinterpret_cast<const uint32_t *>(blk) + r), 0u);
  if (F == 8) return __ldg(reinterpret_cast<const uint2 *>(blk) + r);
  const uint16_t *h = reinterpret_cast<const uint16_t *>(blk + 6 * r);
  return make_uint2((uint32_t)__ldg(h) | ((uint32_t)__ldg(h + 1) << 16), (uint32_t)__ldg(h + 2));
}

// ----------------------------------------------------------------- tiles
struct Phase {
  int phh, phw, Hp, Wp, kh0, kw0, nth, ntw;
  int q0, r0;   // ho = a - u + q0, wo = b - v + r0 for in-phase position (a, b) and tap (u, v)
};

__device__ __forceinline__ Phase get_phase(const ConvParams &p, int ph) {
  Phase q;
  const int s = p.stride;
  q.phh = ph / s;
  q.phw = ph % s;
  q.Hp = q.phh < p.H ? (p.H - q.phh + s - 1) / s : 0;
  q.Wp = q.phw < p.W ? (p.W - q.phw + s - 1) / s : 0;
  q.kh0 = (q.phh + p.pad) % s;
  q.kw0 = (q.phw + p.pad) % s;
  q.nth = q.kh0 < p.Kh ? (p.Kh - q.kh0 + s - 1) / s : 0;
  q.ntw = q.kw0 < p.Kw ? (p.Kw - q.kw0 + s - 1) / s : 0;
  q.q0 = (q.phh + p.pad) / s;
  q.r0 = (q.phw + p.pad) / s;
  return q;
}

struct Tile {
  int m, n, split;   // m: row tile (within its phase for dgrad)
  int nchunks;
  int kg0, kg1;      // wgrad: k-group range of the split
  Phase ph;
};

__device__ __forceinline__ Tile get_tile(const ConvParams &p, int t) {
  Tile T;
  T.n = t % p.n_tiles;
  int rest = t / p.n_tiles;
  T.split = 0;
  T.kg0 = 0;
  T.kg1 = p.kg_total;
  if (p.op == OP_FWD) {
    T.m = rest;
    T.nchunks = (p.kg_total + KCH - 1) / KCH;
  } else if (p.op == OP_WGRAD) {
    T.m = rest % p.m_tiles;
    T.split = rest / p.m_tiles;
    T.kg0 = T.split * p.kg_per_split;
    T.kg1 = min(p.kg_total, T.kg0 + p.kg_per_split);
    T.nchunks = (T.kg1 - T.kg0 + KCH - 1) / KCH;
  } else {
    int m = rest, ph = 0;
    for (;; ++ph) {
      Phase q = get_phase(p, ph);
      const int tiles = (q.Hp * q.Wp * p.NG + 15) / 16;
      if (m < tiles || ph == p.stride * p.stride - 1) {
        T.ph = q;
        break;
      }
      m -= tiles;
    }
    T.m = m;
    T.nchunks = (T.ph.nth * T.ph.ntw * p.COG + KCH - 1) / KCH;
  }
  return T;
}

// ------------------------------------------------------- address tables
// The block feeding core matrix (row group g, k-group k) of operand A, or
// (column group g, k-group k) of operand B, depends on one entry of three
// small tables that the producers rebuild for every chunk: A row groups (16),
// B column groups (BN/8 <= 32) and the chunk's k-groups (KCH).  Combining an
// entry pair is a few integer multiply-adds; v < 0 marks "no block" (padding,
// ragged tail, invalid stride phase): the core matrix is zero.
struct Ent {
  int x, y, z, w, v;
};
struct Tables {
  Ent rg[16];
  Ent cg[32];
  Ent kg[KCH];
};

template <int OP>
__device__ __forceinline__ void fill_tables(const ConvParams &p, const Tile &T, int c, Tables &tb, int tid) {
  Ent e = {0, 0, 0, 0, -1};
  if (tid < 16) {
    const int g = tid;
    if (OP == OP_FWD) {
      const int rg = T.m * 16 + g;
      if (rg < p.Ho * p.Wo * p.NG) {
        const int pos = rg / p.NG, ng = rg - pos * p.NG, ho = pos / p.Wo, wo = pos - ho * p.Wo;
        e = {ho * p.stride - p.pad, wo * p.stride - p.pad, ng, 0, 0};
      }
    } else if (OP == OP_DGRAD) {
      const int rg = T.m * 16 + g;
      if (rg < T.ph.Hp * T.ph.Wp * p.NG) {
        const int pp = rg / p.NG, ng = rg - pp * p.NG, a = pp / T.ph.Wp, b = pp - a * T.ph.Wp;
        e = {a, b, ng, 0, 0};
      }
    } else {
      const int cog = T.m * 16 + g;
      if (cog < p.COG) e = {cog, 0, 0, 0, 0};
    }
    tb.rg[g] = e;
  } else if (tid < 48) {
    const int g = tid - 16;
    if (g < p.BN / 8) {
      const int col = T.n * (p.BN / 8) + g;
      if (OP == OP_FWD) {
        if (col < p.COG) e = {col, 0, 0, 0, 0};
      } else if (OP == OP_DGRAD) {
        if (col < p.CIG) e = {col, 0, 0, 0, 0};
      } else if (col < p.Kh * p.Kw * p.CIG) {
        const int tap = col / p.CIG, cig = col - tap * p.CIG, kh = tap / p.Kw, kw = tap - kh * p.Kw;
        e = {kh, kw, cig, 0, 0};
      }
      tb.cg[g] = e;
    }
  } else if (tid < 48 + KCH) {
    const int k = tid - 48;
    if (OP == OP_FWD) {
      const int kg = c * KCH + k;
      if (kg < p.kg_total) {
        const int tap = kg / p.CIG, cg = kg - tap * p.CIG, kh = tap / p.Kw, kw = tap - kh * p.Kw;
        e = {kh, kw, cg, 0, 0};
      }
    } else if (OP == OP_DGRAD) {
      const int kg = c * KCH + k;
      if (kg < T.ph.nth * T.ph.ntw * p.COG) {
        const int tap = kg / p.COG, cog = kg - tap * p.COG, u = tap / T.ph.ntw, v = tap - u * T.ph.ntw;
        e = {u, v, cog, 0, 0};
      }
    } else {
      const int ka = T.kg0 + c * KCH + k;
      if (ka < T.kg1) {
        const int pos = ka / p.NG, ng = ka - pos * p.NG, ho = pos / p.Wo, wo = pos - ho * p.Wo;
        e = {ho * p.stride - p.pad, wo * p.stride - p.pad, ng, ka, 0};
      }
    }
    tb.kg[k] = e;
  }
}

template <int OP>
__device__ __forceinline__ int64_t a_blk(const ConvParams &p, const Tile &T, const Ent &r, const Ent &k) {
  if ((r.v | k.v) < 0) return -1;
  if (OP == OP_FWD) {
    const int hi = r.x + k.x, wi = r.y + k.y;
    if ((unsigned)hi >= (unsigned)p.H || (unsigned)wi >= (unsigned)p.W) return -1;
    return ((int64_t)(hi * p.W + wi) * p.NG + r.z) * p.CIG + k.z;
  } else if (OP == OP_DGRAD) {
    const int ho = r.x - k.x + T.ph.q0, wo = r.y - k.y + T.ph.r0;
    if ((unsigned)ho >= (unsigned)p.Ho || (unsigned)wo >= (unsigned)p.Wo) return -1;
    return ((int64_t)(ho * p.Wo + wo) * p.NG + r.z) * p.COG + k.z;
  } else {
    return (int64_t)k.w * p.COG + r.x;    // k.w = position * NG + ng
  }
}

template <int OP>
__device__ __forceinline__ int64_t b_blk(const ConvParams &p, const Tile &T, const Ent &c, const Ent &k) {
  if ((c.v | k.v) < 0) return -1;
  if (OP == OP_FWD) {
    return ((int64_t)(k.x * p.Kw + k.y) * p.COG + c.x) * p.CIG + k.z;
  } else if (OP == OP_DGRAD) {
    const int kh = T.ph.kh0 + p.stride * k.x, kw = T.ph.kw0 + p.stride * k.y;
    return ((int64_t)(kh * p.Kw + kw) * p.COG + k.z) * p.CIG + c.x;
  } else {
    const int hi = k.x + c.x, wi = k.y + c.y;
    if ((unsigned)hi >= (unsigned)p.H || (unsigned)wi >= (unsigned)p.W) return -1;
    return ((int64_t)(hi * p.W + wi) * p.NG + k.z) * p.CIG + c.z;
  }
}

// ------------------------------------------------------- requant epilogue
// Requantize one 16-column chunk of a row (thread = one (position, n) row of
// the tile) into two blocks of the packed output (the next layer's
// activations for the forward pass, the lower layer's output gradient for the
// data gradient; nc channels, ncg = nc / 8 groups).  Lanes 8q..8q+7 of a warp
// hold the eight batch rows of one block: the block amax is their shuffle-max.
// TINY: T_scale below 2^-62, encoded from y 2^64 and T_scale 2^64 (s_t is
// then the scaled one; see up64).  RARE: compile the stochastic-rounding
// branch (p.rq.sr; only the out-of-line copy below has it).
template <int F, bool TINY, bool RARE = true>
__device__ __forceinline__ void requant_chunk(const ConvParams &p, const float (&y)[16], int pos, int ng, int n_in,
                                              int co0, bool row_ok, float s_t, float s_true, int nc, int ncg,
                                              uint32_t &amax_acc) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int co = co0 + 8 * h;
    float v[8], v_true[8];
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      m = max(m, __float_as_uint(y[8 * h + j]) & 0x7FFFFFFFu);
      v_true[j] = y[8 * h + j];
      v[j] = TINY ? up64(y[8 * h + j]) : y[8 * h + j];
    }
    if (!row_ok) m = 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    amax_acc = max(amax_acc, m);
    if (!row_ok || co >= nc) continue;
    const uint32_t bsc = block_scale_code<F>(TINY ? up64(__uint_as_float(m)) : __uint_as_float(m), s_t);
    const float bs = code_value<8>(bsc);
    const int64_t blk = ((int64_t)pos * p.NG + ng) * ncg + co / 8;
    // stochastic codes (MicroQonv §III-A, see encode_row8_sr) from the unscaled T_scale s_true
    const uint64_t bits = RARE && p.rq.sr ? encode_row8_sr<F>(v_true, __fmul_rn(bs, s_true), p.rq.sr_seed, blk, n_in)
                                          : encode_row8<F>(v, bs, s_t);
    uint8_t *dst = p.rq.codes + blk * Fmt<F>::BLOCK_BYTES;
    if (F == 4) {
      reinterpret_cast<uint32_t *>(dst)[n_in] = (uint32_t)bits;
    } else if (F == 6) {
      uint16_t *d16 = reinterpret_cast<uint16_t *>(dst + 6 * n_in);
      d16[0] = (uint16_t)bits;
      d16[1] = (uint16_t)(bits >> 16);
      d16[2] = (uint16_t)(bits >> 32);
    } else {
      reinterpret_cast<uint64_t *>(dst)[n_in] = bits;
    }
    if (n_in == 0) p.rq.scales[blk] = (uint8_t)bsc;
  }
}

// The tiny-T_scale and stochastic requantizations, kept out of line (rare;
// inlined they would raise the register pressure of every requantizing kernel).
template <int F>
__device__ __noinline__ void requant_chunk_rare(const ConvParams &p, const float (&y)[16], int pos, int ng, int n_in,
                                                int co0, bool row_ok, float s_t, float s_true, int nc, int ncg,
                                                bool tiny, uint32_t &amax_acc) {
  if (tiny) requant_chunk<F, true>(p, y, pos, ng, n_in, co0, row_ok, s_t, s_true, nc, ncg, amax_acc);
  else requant_chunk<F, false>(p, y, pos, ng, n_in, co0, row_ok, s_t, s_true, nc, ncg, amax_acc);
}

// --------------------------------------------------------------- kernel
struct SmemCtl {
  Tables tab[2];
  volatile int prod_ok[2];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t done;
  uint32_t tmem_base;
  volatile int abort_flag;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, const ConvParams &p, SmemCtl *ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 127u) == 127u) {
      if (ctl->abort_flag) return false;
      if (globaltimer_ns() - t0 > 2000000000ull) {
        atomicOr(p.status, ST_TIMEOUT);
        ctl->abort_flag = 1;
        return false;
      }
    }
  }
}

template <int OP, int FA, int FB, int FR>
__global__ void __launch_bounds__(CONV_THREADS, 1) conv_kernel(const ConvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_stage = p.BN * 128;                    // (BN/8) x KCH core matrices
  uint8_t *a_ring = smem;
  uint8_t *b_ring = smem + STAGES * A_STAGE;
  SmemCtl *ctl = reinterpret_cast<SmemCtl *>(b_ring + STAGES * b_stage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.m_tiles * p.n_tiles * p.k_splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], PROD_WARPS * 32);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->acc_full[b], 1);
      mbar_init(&ctl->acc_empty[b], EPI_WARPS * 32);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) tmem_alloc(&ctl->tmem_base, 2 * p.acc_stride);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp < PROD_WARPS) {
    // ------------------------------------------------------ producers
    // Every thread first issues all loads of its (up to MAXJ) core-matrix
    // rows for the stage, then decodes and stores them: the global latency of
    // one stage overlaps instead of serialising row by row.  Stage layout:
    // core matrix (group g, k-group k) at (g * KCH + k) * 128 bytes.
    constexpr int MAXJ = 4 + 8;                       // 4 A rows + up to 8 B rows per thread
    const int ptid = threadIdx.x;
    const int btasks = p.BN * 8;
    int it = 0;
    bool run = true;
    for (int t = blockIdx.x; t < num_tiles && run; t += gridDim.x) {
      const Tile T = get_tile(p, t);
      for (int c = 0; c < T.nchunks; ++c, ++it) {
        const int s = it % STAGES;
        Tables &tb = ctl->tab[it & 1];
        if (ptid == 0) ctl->prod_ok[it & 1] = wait_or_abort(&ctl->empty[s], ((it / STAGES) & 1) ^ 1, p, ctl) ? 1 : 0;
        fill_tables<OP>(p, T, c, tb, ptid);
        asm volatile("bar.sync 1, %0;" ::"n"(PROD_WARPS * 32) : "memory");
        if (!ctl->prod_ok[it & 1]) { run = false; break; }
        uint8_t *sa = a_ring + s * A_STAGE, *sb = b_ring + s * b_stage;
        uint2 raw[MAXJ];
        uint32_t scb[MAXJ];
        bool ok[MAXJ];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = ptid + PROD_WARPS * 32 * j, cm = i >> 3, r = i & 7;
          const int64_t blk = a_blk<OP>(p, T, tb.rg[cm >> 3], tb.kg[cm & 7]);
          ok[j] = blk >= 0;
          if (ok[j]) {
            raw[j] = load_raw<FA>(p.a.codes + blk * Fmt<FA>::BLOCK_BYTES, r);
            scb[j] = __ldg(p.a.scales + blk);
          }
        }
#pragma unroll
        for (int j = 4; j < MAXJ; ++j) {
          const int i = ptid + PROD_WARPS * 32 * (j - 4), cm = i >> 3, r = i & 7;
          ok[j] = false;
          if (i < btasks) {
            const int64_t blk = b_blk<OP>(p, T, tb.cg[cm >> 3], tb.kg[cm & 7]);
            ok[j] = blk >= 0;
            if (ok[j]) {
              raw[j] = load_raw<FB>(p.b.codes + blk * Fmt<FB>::BLOCK_BYTES, r);
              scb[j] = __ldg(p.b.scales + blk);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = ptid + PROD_WARPS * 32 * j;
          const uint4 v = ok[j] ? decode_raw<FA>(raw[j], scale_pair<FA>((uint8_t)scb[j])) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(sa + i * 16) = v;
        }
#pragma unroll
        for (int j = 4; j < MAXJ; ++j) {
          const int i = ptid + PROD_WARPS * 32 * (j - 4);
          if (i < btasks) {
            const uint4 v = ok[j] ? decode_raw<FB>(raw[j], scale_pair<FB>((uint8_t)scb[j])) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(sb + i * 16) = v;
          }
        }
        fence_async_smem();
        mbar_arrive(&ctl->full[s]);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr bool a_mn = (OP == OP_WGRAD);
      constexpr bool b_mn = (OP != OP_FWD);
      const uint32_t idesc = idesc_f16(128, p.BN, a_mn, b_mn);
      constexpr uint32_t lbo = 128, sbo = KCH * 128;   // core matrix (g, k) at (g * KCH + k) * 128
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tc) {
        const Tile T = get_tile(p, t);
        const int buf = tc & 1;
        if (!wait_or_abort(&ctl->acc_empty[buf], ((tc >> 1) & 1) ^ 1, p, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * p.acc_stride;
        for (int c = 0; c < T.nchunks; ++c, ++it) {
          const int s = it % STAGES;
          if (!wait_or_abort(&ctl->full[s], (it / STAGES) & 1, p, ctl)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(a_ring + s * A_STAGE), sb = smem_u32(b_ring + s * b_stage);
#pragma unroll
          for (int kk = 0; kk < KCH / 2; ++kk) {
            const uint64_t da = sdesc(sa + kk * 2 * lbo, lbo, sbo);
            const uint64_t db = sdesc(sb + kk * 2 * lbo, lbo, sbo);
            umma_f16(d, da, db, idesc, (c > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&ctl->empty[s]);
        }
        if (!ok) break;
        umma_commit(&ctl->acc_full[buf]);
      }
      // every MMA issued above has completed once `done` flips
      umma_commit(&ctl->done);
      // every MMA issued so far completes before the TMEM is freed, whatever the abort flag says
      mbar_wait(&ctl->done, 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue
    const int ew = warp - PROD_WARPS;           // TMEM lanes 32*ew .. 32*ew+31
    const int row = ew * 32 + lane;
    const float pre = p.pre_mult;
    const float f = (*p.a.s_t) * (*p.b.s_t) * pre;
    float rq_st = 0.0f;
    if (FR) rq_st = __fdiv_rn(*p.rq.amax_in, Fmt<FR ? FR : 4>::DENOM);
    const bool rq_tiny = FR && is_tiny_scale(rq_st);
    const float rq_stq = rq_tiny ? rq_st * TINY_MULT : rq_st;   // the T_scale quotients are formed with
    uint32_t amax_acc = 0;
    int tc = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tc) {
      const Tile T = get_tile(p, t);
      const int buf = tc & 1;
      if (!wait_or_abort(&ctl->acc_full[buf], (tc >> 1) & 1, p, ctl)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + buf * p.acc_stride + ((uint32_t)(ew * 32) << 16);

      // where this row goes
      int64_t obase = -1;
      int pos = 0, ng = 0, n_in = row & 7;
      if (OP == OP_FWD) {
        const int rg = T.m * 16 + (row >> 3);
        if (rg < p.Ho * p.Wo * p.NG) {
          pos = rg / p.NG;
          ng = rg - pos * p.NG;
          obase = ((int64_t)pos * p.Cout) * p.N + ng * 8 + n_in;
        }
      } else if (OP == OP_DGRAD) {
        const int rg = T.m * 16 + (row >> 3);
        if (rg < T.ph.Hp * T.ph.Wp * p.NG) {
          const int pp = rg / p.NG;
          ng = rg - pp * p.NG;
          const int a = pp / T.ph.Wp, b = pp - a * T.ph.Wp;
          const int hi = T.ph.phh + p.stride * a, wi = T.ph.phw + p.stride * b;
          pos = hi * p.W + wi;
          obase = ((int64_t)pos * p.Cin) * p.N + ng * 8 + n_in;
        }
      } else {
        const int co = T.m * 128 + row;
        if (co < p.Cout) obase = ((int64_t)T.split * p.Cout + co) * p.ncols;
      }
      const int col0 = T.n * p.BN;
      const int ncol_valid = OP == OP_FWD ? p.Cout : OP == OP_DGRAD ? p.Cin : p.ncols;

      for (int c0 = 0; c0 < p.BN; c0 += 16) {
        uint32_t r[16];
        if (T.nchunks > 0) {
          tmem_ld16(tbase + c0, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = 0u;
        }
        float y[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] = __uint_as_float(r[j]) * (OP == OP_WGRAD ? 1.0f : f);
        if (OP == OP_WGRAD) {
          if (obase >= 0) {
            float *o = p.out + obase + col0 + c0;
            if (col0 + c0 + 16 <= ncol_valid) {
#pragma unroll
              for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4 *>(o + j) = make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]);
            } else {
              for (int j = 0; j < 16; ++j)
                if (col0 + c0 + j < ncol_valid) o[j] = y[j];
            }
          }
        } else {
          if (obase >= 0 && p.out) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (col0 + c0 + j < ncol_valid) p.out[obase + (int64_t)(col0 + c0 + j) * p.N] = y[j];
          }
          if (FR) {
            const int nc = OP == OP_FWD ? p.Cout : p.Cin;
            if (rq_tiny || p.rq.sr)
              requant_chunk_rare<FR ? FR : 4>(p, y, pos, ng, n_in, col0 + c0, obase >= 0, rq_stq, rq_st, nc,
                                              nc / 8, rq_tiny, amax_acc);
            else
              requant_chunk<FR ? FR : 4, false, false>(p, y, pos, ng, n_in, col0 + c0, obase >= 0, rq_stq, rq_st,
                                                       nc, nc / 8, amax_acc);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->acc_empty[buf]);
    }
    if (FR && OP != OP_WGRAD) {
#pragma unroll
      for (int o = 16; o; o >>= 1) amax_acc = max(amax_acc, __shfl_xor_sync(0xFFFFFFFFu, amax_acc, o));
      if (lane == 0 && amax_acc && p.rq.amax_out_bits) atomicMax(p.rq.amax_out_bits, amax_acc);
      if (blockIdx.x == 0 && threadIdx.x == PROD_WARPS * 32) *p.rq.s_t_out = rq_st;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) tmem_dealloc(tmem, 2 * p.acc_stride);
}

// ------------------------------------------------------- wgrad reduction
// dW[co][ci][kh][kw] = f * sum_split partial[split][co][(kh*Kw+kw)*Cin + ci],
// summed in split order (deterministic).
__global__ void wgrad_reduce_kernel(const ConvParams p, float *__restrict__ dw) {
  const int64_t total = (int64_t)p.Cout * p.ncols;
  const float f = (*p.a.s_t) * (*p.b.s_t) * p.pre_mult;
  const int KK = p.Kh * p.Kw;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int k = 0; k < p.k_splits; ++k) s += p.out[(int64_t)k * total + i];
    const int64_t co = i / p.ncols;
    const int col = (int)(i - co * p.ncols);
    const int tap = col / p.Cin, ci = col - tap * p.Cin;
    dw[(co * p.Cin + ci) * KK + tap] = s * f;
  }
}

// ------------------------------------------------------------------ host
static int round_up(int x, int m) { return (x + m - 1) / m * m; }
static int pow2_at_least(int x) {
  int v = 32;
  while (v < x) v <<= 1;
  return v;
}

int64_t conv_plan(ConvParams &p) {
  const int KK = p.Kh * p.Kw;
  if (p.op == OP_FWD) {
    p.BN = std::min(256, round_up(p.Cout, 16));
    p.n_tiles = (p.Cout + p.BN - 1) / p.BN;
    p.m_tiles = (p.Ho * p.Wo * p.NG + 15) / 16;
    p.k_splits = 1;
    p.kg_total = KK * p.CIG;
  } else if (p.op == OP_DGRAD) {
    p.BN = std::min(256, round_up(p.Cin, 16));
    p.n_tiles = (p.Cin + p.BN - 1) / p.BN;
    int m = 0;
    const int s = p.stride;
    for (int ph = 0; ph < s * s; ++ph) {
      const int phh = ph / s, phw = ph % s;
      const int Hp = phh < p.H ? (p.H - phh + s - 1) / s : 0, Wp = phw < p.W ? (p.W - phw + s - 1) / s : 0;
      m += (Hp * Wp * p.NG + 15) / 16;
    }
    p.m_tiles = m;
    p.k_splits = 1;
    p.kg_total = 0;
  } else {
    p.ncols = KK * p.Cin;
    p.BN = std::min(256, round_up(p.ncols, 16));
    p.n_tiles = (p.ncols + p.BN - 1) / p.BN;
    p.m_tiles = (p.Cout + 127) / 128;
    p.kg_total = p.Ho * p.Wo * p.NG;
    const int mn = p.m_tiles * p.n_tiles;
    int splits = std::max(1, (296 + mn - 1) / mn);
    splits = std::min(splits, std::max(1, p.kg_total / (4 * KCH)));
    p.kg_per_split = round_up((p.kg_total + splits - 1) / splits, KCH);
    p.k_splits = (p.kg_total + p.kg_per_split - 1) / p.kg_per_split;
    p.wg_rows = round_up(p.Cout, 128);
  }
  p.acc_stride = pow2_at_least(p.BN);
  return (int64_t)p.m_tiles * p.n_tiles * p.k_splits;
}

size_t conv_smem_bytes(const ConvParams &p) {
  return 1024 + (size_t)STAGES * (A_STAGE + p.BN * 128) + sizeof(SmemCtl);
}

template <int OP, int FA, int FB, int FR>
static cudaError_t launch_one(const ConvParams &p, int grid, size_t smem, cudaStream_t s) {
  auto k = conv_kernel<OP, FA, FB, FR>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, CONV_THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

template <int OP, int F, int FR>
static cudaError_t dispatch_b(const ConvParams &p, int grid, size_t smem, cudaStream_t s) {
  switch (p.b.fmt) {
    case 4: return launch_one<OP, F, 4, FR>(p, grid, smem, s);
    case 6: return launch_one<OP, F, 6, FR>(p, grid, smem, s);
    default: return launch_one<OP, F, 8, FR>(p, grid, smem, s);
  }
}

template <int OP, int FR>
static cudaError_t dispatch_a(const ConvParams &p, int grid, size_t smem, cudaStream_t s) {
  switch (p.a.fmt) {
    case 4: return dispatch_b<OP, 4, FR>(p, grid, smem, s);
    case 6: return dispatch_b<OP, 6, FR>(p, grid, smem, s);
    default: return dispatch_b<OP, 8, FR>(p, grid, smem, s);
  }
}

cudaError_t launch_conv(const ConvParams &p, int num_sms, cudaStream_t s) {
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles * p.k_splits;
  if (tiles <= 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>(tiles, num_sms);
  const size_t smem = conv_smem_bytes(p);
  if (p.op == OP_FWD) {
    if (p.rq.codes) {
      switch (p.rq.fmt) {
        case 4: return dispatch_a<OP_FWD, 4>(p, grid, smem, s);
        case 6: return dispatch_a<OP_FWD, 6>(p, grid, smem, s);
        default: return dispatch_a<OP_FWD, 8>(p, grid, smem, s);
      }
    }
    return dispatch_a<OP_FWD, 0>(p, grid, smem, s);
  }
  if (p.op == OP_DGRAD) {
    if (p.rq.codes) {
      switch (p.rq.fmt) {
        case 4: return dispatch_a<OP_DGRAD, 4>(p, grid, smem, s);
        case 6: return dispatch_a<OP_DGRAD, 6>(p, grid, smem, s);
        default: return dispatch_a<OP_DGRAD, 8>(p, grid, smem, s);
      }
    }
    return dispatch_a<OP_DGRAD, 0>(p, grid, smem, s);
  }
  return dispatch_a<OP_WGRAD, 0>(p, grid, smem, s);
}

cudaError_t launch_wgrad_reduce(const ConvParams &p, float *dw, cudaStream_t s) {
  const int64_t total = (int64_t)p.Cout * p.ncols;
  const int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
  wgrad_reduce_kernel<<<grid, 256, 0, s>>>(p, dw);
  return cudaGetLastError();
}

}  // namespace mq
