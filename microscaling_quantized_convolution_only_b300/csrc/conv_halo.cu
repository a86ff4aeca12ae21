// conv_halo.cu -- the halo-reuse weight-gradient kernel, and the host side
// of the halo kernels: tensor maps, tile planners and launches.  The
// forward and data-gradient kernel lives in conv_halo.cuh (instantiated by
// conv_halo_fwd.cu and conv_halo_dgrad.cu); its design notes are there.
#include <algorithm>
#include <cstring>
#include <numeric>
#include <mutex>

#include "conv_halo.cuh"

namespace mq {

// ---------------------------------------------------------------- wgrad
// G_W[co][kh][kw][ci] = sum over (ho, wo, n) of dY[ho][wo][co][n] *
// X[ho + kh - pad][wo + kw - pad][ci][n]  (MicroQonv §IV-A: G_W = G_Y X'^T).
// A CTA tile fixes kh, a block of 128 output channels and BNc input channels
// and walks a range of chunks; a chunk is one output row ho, P positions and
// G batch groups (K = 8 P G).  Per chunk it stages the dY blocks (P x G x 16
// channel groups) and the one-row X halo (P + Kw - 1 positions) and decodes
// both once; tap kw reads the halo through a descriptor shifted by kw
// positions.  Accumulator kw (128 x BNc fp32) sits at TMEM column kw * acc.
// Both operands are MN-major: a block row is 8 channels of one batch element.
// warp roles of the weight-gradient kernel: ten decoders (its two operands
// are both decoded per chunk), eight epilogue warps, the TMA / scale
// producer and the MMA issuer
constexpr int WG_DEC_WARPS = 10;
constexpr int WG_DEC_THREADS = WG_DEC_WARPS * 32;
constexpr int WG_EPI_WARP0 = 10;
constexpr int WG_EPI_WARPS = 8;
constexpr int WG_TMA_WARP = 18;
constexpr int WG_MMA_WARP = 19;
constexpr int WG_THREADS = 20 * 32;

struct WgCtl {
  uint64_t pfull[MAX_PS], pempty[MAX_PS];
  uint64_t dfull[DSTAGES], dempty[DSTAGES];
  uint64_t acc_full, acc_empty;
  uint64_t done;
  uint32_t tmem_base;
  volatile int abort_flag;
};

struct WgTile {
  int kh, c0, m0, split, q0, q1;   // kernel row, first input / output channel, split, chunk range
};

__device__ __forceinline__ WgTile wg_tile(const HaloWgrad &p, int t) {
  WgTile w;
  int r = t;
  w.kh = r % p.Kh;
  r /= p.Kh;
  w.c0 = (r % p.c_tiles) * p.BNc;
  r /= p.c_tiles;
  w.m0 = (r % p.m_tiles) * 128;
  w.split = r / p.m_tiles;
  w.q0 = w.split * p.chunks_per_split;
  w.q1 = min(p.total_chunks, w.q0 + p.chunks_per_split);
  return w;
}

// bounded wait, as hc_wait
__device__ __forceinline__ bool wg_wait(uint64_t *bar, uint32_t parity, const HaloWgrad &p, WgCtl *ctl) {
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

template <int FA, int FB>
__global__ void __launch_bounds__(WG_THREADS, 1)
    halo_wgrad_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const HaloWgrad p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  WgCtl *ctl = reinterpret_cast<WgCtl *>(smem + p.off_ctl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int BBA = Fmt<FA>::BLOCK_BYTES, BBB = Fmt<FB>::BLOCK_BYTES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.PS; ++s) {
      mbar_init(&ctl->pfull[s], 64);
      mbar_init(&ctl->pempty[s], WG_DEC_WARPS);
    }
    for (int s = 0; s < DSTAGES; ++s) {
      mbar_init(&ctl->dfull[s], WG_DEC_WARPS);
      mbar_init(&ctl->dempty[s], 1);
    }
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->acc_empty, WG_EPI_WARPS);
    mbar_init(&ctl->done, 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == WG_MMA_WARP) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == WG_TMA_WARP) {
    // ----------------------------------------------------------- producer
    // lane 0 issues the two code boxes, all lanes copy the chunk's block
    // scales asynchronously (zero where the block is out of range); 64
    // arrivals (two per lane) + the box bytes complete a stage.
    int pit = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const WgTile T = wg_tile(p, t);
      for (int q = T.q0; q < T.q1; ++q, ++pit) {
        const int ps = pit % p.PS;
        int okw = 1;
        if (lane == 0) okw = wg_wait(&ctl->pempty[ps], ((pit / p.PS) & 1) ^ 1, p, ctl) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, okw, 0)) { ok = false; break; }
        const int gb = q % p.tiles_g, rest = q / p.tiles_g;
        const int g0 = gb * p.G, wo0 = (rest % p.tiles_w) * p.P, ho = rest / p.tiles_w;
        const int hi = p.S * ho + T.kh - p.pad;
        uint8_t *stage = smem + p.off_pk + ps * p.pk_stage;
        uint8_t *sc = stage + p.pk_sc_off;
        if (lane == 0) {
          mbar_add_tx(&ctl->pfull[ps], p.pk_bytes);
          tma_load_4d(stage, &tm_a, &ctl->pfull[ps], (T.m0 / 8) * BBA / 8, g0, wo0, ho);
          if (p.S == 1) {
            tma_load_4d(stage + p.pk_b_off, &tm_b, &ctl->pfull[ps], (T.c0 / 8) * BBB / 8, g0, wo0 - p.pad, hi);
          } else {
            // stride 2: X halo phase ph = input columns 2 wo0 - pad + ph + 2 k
            const uint32_t ph_bytes = (uint32_t)(p.PHP * p.G * p.CB * BBB);   // a multiple of 128
            for (int ph = 0; ph < p.NPH; ++ph) {
              const int wc0 = 2 * wo0 - p.pad + ph, gph = wc0 & 1;
              tma_load_5d(stage + p.pk_b_off + ph * ph_bytes, &tm_b, &ctl->pfull[ps], (T.c0 / 8) * BBB / 8, g0, gph,
                          (wc0 - gph) / 2, hi);
            }
          }
        }
        // dY block scales: run (p, j) = 16 output-channel groups
        const int mbv = min(16, p.COG - T.m0 / 8);
        copy_runs_rt(
            p.gran_a, sc, p.KG, 16, 16,
            [&](int r) -> const uint8_t * {
              const int pp = r / p.G, j = r - pp * p.G, wo = wo0 + pp;
              if (wo >= p.Wo) return nullptr;
              return p.a_scales + (((int64_t)ho * p.Wo + wo) * p.NG + g0 + j) * p.COG + T.m0 / 8;
            },
            [&](int) { return mbv; }, p.a_scales, lane);
        // X halo block scales: run (phase, wc, j) = CB input-channel groups;
        // the padding positions at the end of a phase get zeros
        const int cbv = min(p.CB, p.CIG - T.c0 / 8), ph_runs = p.PHP * p.G;
        copy_runs_rt(
            p.gran_b, sc + p.na_blocks, p.NPH * ph_runs, p.CB, p.CB,
            [&](int r) -> const uint8_t * {
              const int ph = r / ph_runs, rr = r - ph * ph_runs;
              const int wc = rr / p.G, j = rr - wc * p.G, wi = p.S * wo0 - p.pad + ph + p.S * wc;
              if (wc >= p.WP) return nullptr;
              if ((unsigned)hi >= (unsigned)p.H || (unsigned)wi >= (unsigned)p.W) return nullptr;
              return p.b_scales + (((int64_t)hi * p.W + wi) * p.NG + g0 + j) * p.CIG + T.c0 / 8;
            },
            [&](int) { return cbv; }, p.b_scales, lane);
        cp_async_arrive(&ctl->pfull[ps]);
        mbar_arrive(&ctl->pfull[ps]);
      }
    }
    // the copies in flight (boxes and every lane's scale copies) land before exit
    if (lane == 0) {
      for (int i = 0; i < p.PS && i < pit; ++i) {
        const int q = pit - 1 - i;
        hc_drain(&ctl->pfull[q % p.PS], (q / p.PS) & 1, p.status);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else if (warp < WG_DEC_WARPS) {
    // ------------------------------------------------------------ decoders
    const int tid = threadIdx.x;
    int pit = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const WgTile T = wg_tile(p, t);
      for (int q = T.q0; q < T.q1; ++q, ++pit) {
        const int ps = pit % p.PS, ds = pit % DSTAGES;
        if (!wg_wait(&ctl->pfull[ps], (pit / p.PS) & 1, p, ctl)) { ok = false; break; }
        if (!wg_wait(&ctl->dempty[ds], ((pit / DSTAGES) & 1) ^ 1, p, ctl)) { ok = false; break; }
        const uint8_t *pk = smem + p.off_pk + ps * p.pk_stage;
        const uint8_t *sc = pk + p.pk_sc_off;
        uint8_t *dec = smem + p.off_dec + ds * p.dec_stage;
        const int na = p.na_blocks * 8;
        for (int i = tid; i < na; i += WG_DEC_THREADS) {
          const int blk = i >> 3, r = i & 7;
          const uint4 v = decode_raw<FA>(row8_bits<FA>(pk + blk * BBA, r), scale_pair<FA>(sc[blk]));
          *reinterpret_cast<uint4 *>(dec + i * 16) = v;
        }
        const int nb = p.nb_blocks * 8;
        const uint8_t *pkb = pk + p.pk_b_off;
        uint8_t *decb = dec + p.dec_b_off;
        for (int i = tid; i < nb; i += WG_DEC_THREADS) {
          const int blk = i >> 3, r = i & 7;
          const uint4 v = decode_raw<FB>(row8_bits<FB>(pkb + blk * BBB, r), scale_pair<FB>(sc[p.na_blocks + blk]));
          *reinterpret_cast<uint4 *>(decb + i * 16) = v;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl->pempty[ps]);
          mbar_arrive(&ctl->dfull[ds]);
        }
      }
    }
  } else if (warp == WG_MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, p.BNc, true, true);
      const uint32_t a_lbo = 16 * 128, b_lbo = (uint32_t)p.CB * 128;
      // descriptor low words stepped by (bytes >> 4), see the halo kernel
      const uint64_t a_desc = sdesc(smem_u32(smem + p.off_dec), a_lbo, 128);
      const uint64_t b_desc = sdesc(smem_u32(smem + p.off_dec + p.dec_b_off), b_lbo, 128);
      const uint32_t a_hi = (uint32_t)(a_desc >> 32), b_hi = (uint32_t)(b_desc >> 32);
      const uint32_t d_stage = p.dec_stage >> 4;
      const uint32_t a_kk = (2 * a_lbo) >> 4, b_kk = (2 * b_lbo) >> 4;   // 16 more K (two k-groups)
      const uint32_t b_kw = (uint32_t)((p.G * p.CB * 128) >> 4);             // one halo position
      const uint32_t b_phase = (uint32_t)((p.PHP * p.G * p.CB * 128) >> 4);  // one column phase
      const int sh = p.S - 1;   // tap kw: column phase kw & sh, kw >> sh positions in
      constexpr int KK = 8;     // MMAs per tap and chunk: K = 8 P G = 128 (KG = 16)
      int pit = 0, k = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++k) {
        const WgTile T = wg_tile(p, t);
        if (!wg_wait(&ctl->acc_empty, (k & 1) ^ 1, p, ctl)) break;
        tc_fence_after();
        for (int q = T.q0; q < T.q1; ++q, ++pit) {
          const int ds = pit % DSTAGES;
          if (!wg_wait(&ctl->dfull[ds], (pit / DSTAGES) & 1, p, ctl)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_stage = (uint32_t)a_desc + (uint32_t)ds * d_stage;
          const uint32_t b_stage = (uint32_t)b_desc + (uint32_t)ds * d_stage;
          for (int kw = 0; kw < p.Kw; ++kw) {
            const uint32_t d = tmem + kw * p.acc_cols;
            const uint32_t b_w = b_stage + (uint32_t)(kw & sh) * b_phase + (uint32_t)(kw >> sh) * b_kw;
            umma_f16(d, desc_of(a_hi, a_stage), desc_of(b_hi, b_w), idesc, q > T.q0 ? 1u : 0u);
#pragma unroll
            for (int kk = 1; kk < KK; ++kk)
              umma_f16_acc(d, desc_of(a_hi, a_stage + kk * a_kk), desc_of(b_hi, b_w + kk * b_kk), idesc);
          }
          umma_commit(&ctl->dempty[ds]);
        }
        if (!ok) break;
        umma_commit(&ctl->acc_full);
      }
      umma_commit(&ctl->done);
      hc_drain(&ctl->done, 0, p.status);   // every MMA issued so far has completed
    }
    __syncwarp();
  } else if (warp >= WG_EPI_WARP0 && warp < WG_EPI_WARP0 + WG_EPI_WARPS) {
    // ------------------------------------------------------------- epilogue
    const int qd = warp & 3;
    const int half = (warp - WG_EPI_WARP0) >> 2;
    const int row = qd * 32 + lane;
    int k = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++k) {
      const WgTile T = wg_tile(p, t);
      if (!wg_wait(&ctl->acc_full, k & 1, p, ctl)) break;
      tc_fence_after();
      const int co = T.m0 + row;
      float *orow = p.out + ((int64_t)T.split * p.Cout + co) * p.ncols + (int64_t)T.kh * p.Kw * p.Cin + T.c0;
      for (int kw = 0; kw < p.Kw; ++kw) {
        const uint32_t tb = tmem + kw * p.acc_cols + ((uint32_t)(qd * 32) << 16);
        for (int c = 16 * half; c < p.BNc; c += 32) {
          uint32_t r[16];
          tmem_ld16(tb + c, r);
          tmem_wait_ld();
          if (co < p.Cout) {
            float *o = orow + kw * p.Cin + c;
            if (T.c0 + c + 16 <= p.Cin) {
#pragma unroll
              for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4 *>(o + jj) = make_float4(__uint_as_float(r[jj]), __uint_as_float(r[jj + 1]),
                                                                  __uint_as_float(r[jj + 2]), __uint_as_float(r[jj + 3]));
            } else {
              for (int jj = 0; jj < 16; ++jj)
                if (T.c0 + c + jj < p.Cin) o[jj] = __uint_as_float(r[jj]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == WG_MMA_WARP) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

// Row-major tensor of `rank` dims (dims[0] innermost, in elements of `esize`
// bytes), box `box`, no swizzle, zero fill out of range.  `map` points to a
// 64-byte aligned CUtensorMap.
bool make_tensor_map(void *map, const void *base, int esize, int rank, const uint64_t *dims, const uint32_t *box) {
  uint64_t gs[4];
  uint64_t stride = (uint64_t)esize;
  for (int i = 0; i < rank; ++i) {
    if (i > 0) gs[i - 1] = stride;
    stride *= dims[i];
  }
  return make_tensor_map_strided(map, base, esize, rank, dims, gs, box);
}

bool make_tensor_map_strided(void *map, const void *base, int esize, int rank, const uint64_t *dims,
                             const uint64_t *strides, const uint32_t *box) {
  auto fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bd[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
    es[i] = 1;
    if (i > 0) gs[i - 1] = strides[i - 1];
  }
  const CUtensorMapDataType dt = esize == 8 ? CU_TENSOR_MAP_DATA_TYPE_UINT64
                                 : esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                 : esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                              : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(static_cast<CUtensorMap *>(map), dt, (cuuint32_t)rank, const_cast<void *>(base), gd, gs, bd, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr size_t SMEM_LIMIT = 227 * 1024;

size_t halo_smem(HaloConv &h, int bba, int bbb) {
  const int taps = h.Kh * h.Kw;
  // stride 2: the halo's even and odd input columns are staged as two
  // phases, so tap v reads phase v % 2 from position v / 2 on
  h.WP = h.S == 1 ? h.P + h.HKw - 1 : h.P + (h.HKw - 1) / 2;
  h.NPH = (h.S == 2 && h.Kw > 1) ? 2 : 1;
  h.RH = h.S * (h.R - 1) + h.HKh;
  h.PHP = h.RH * h.WP;
  if (h.NPH > 1)   // each phase's packed box must start 128-byte aligned
    while ((h.PHP * h.G * CGC * bba) % 128) ++h.PHP;
  h.nh_blocks = h.NPH * h.PHP * h.G * CGC;
  h.nb_blocks = taps * h.NB * CGC;
  h.dec_b_off = (uint32_t)h.nh_blocks * 128;
  h.dec_stage = (uint32_t)(h.nh_blocks + h.nb_blocks) * 128;
  h.pk_b_off = (uint32_t)((h.nh_blocks * bba + 127) / 128 * 128);
  // with the decoded weight copy the packed stages hold the halo only, and the
  // weights go by TMA straight into the decoded stages (wd_bytes per chunk)
  const int nbp = h.wd ? 0 : h.nb_blocks;
  h.wd_bytes = h.wd ? (uint32_t)h.nb_blocks * 128 : 0u;
  // bytes the boxes deliver per chunk (the phase padding is not written)
  h.pk_bytes = (uint32_t)(h.NPH * h.RH * h.WP * h.G * CGC * bba + nbp * bbb);
  h.pk_stage = (uint32_t)((h.pk_b_off + nbp * bbb + 127) / 128 * 128);
  h.sc_bytes = (uint32_t)(h.NPH * h.PHP * h.G * h.CGin);
  h.scw_off = (h.sc_bytes + 15) / 16 * 16;
  const uint32_t scw = h.wd ? 0u : h.op == OP_FWD ? (uint32_t)(taps * h.NB * h.CIG) : (uint32_t)(taps * h.COG * h.NB);
  h.sc_stride = (h.scw_off + scw + 127) / 128 * 128;
  const size_t fixed = 1024 + (size_t)DSTAGES * h.dec_stage + 2 * h.sc_stride + sizeof(HcCtl) + 128;
  if (fixed + 2 * (size_t)h.pk_stage > SMEM_LIMIT) return 0;
  h.PS = (int)std::min<size_t>(MAX_PS, (SMEM_LIMIT - fixed) / h.pk_stage);
  h.off_dec = 0;
  h.off_pk = DSTAGES * h.dec_stage;
  h.off_sc = h.off_pk + h.PS * h.pk_stage;
  h.off_ctl = h.off_sc + 2 * h.sc_stride;
  return 1024 + (size_t)h.off_ctl + sizeof(HcCtl);
}

// largest power of two dividing x, at most 16 (the cp.async granule)
int pow2_part(int x) {
  int g = 1;
  while (g < 16 && x % (2 * g) == 0) g *= 2;
  return g;
}

int pow2_at_least32(int x) {
  int v = 32;
  while (v < x) v <<= 1;
  return v;
}

}  // namespace

// Plans the halo kernel for a forward (stride 1 or 2) or data-gradient
// (stride 1, or stride 2 as output quads) convolution;
// returns false when the layer does not fit its constraints (the caller then
// uses the generic kernel).
bool halo_plan(const ConvParams &cp, HaloConv &h, int num_sms) {
  std::memset(&h, 0, sizeof(h));
  if (cp.op != OP_FWD && cp.op != OP_DGRAD) return false;
  // stride-2 forward reads the input through a [H][W/2][2] view; the
  // stride-2 data gradient runs as output quads (all four phases per tile)
  const bool qd = cp.op == OP_DGRAD && cp.stride == 2;
  if (cp.stride != 1 && !(cp.stride == 2 && cp.op == OP_FWD && cp.W % 2 == 0) && !qd) return false;
  h.op = cp.op;
  h.S = qd ? 1 : cp.stride;
  h.N = cp.N;
  h.NG = cp.NG;
  h.Kh = cp.Kh;
  h.Kw = cp.Kw;
  h.COG = cp.COG;
  h.CIG = cp.CIG;
  if (cp.op == OP_FWD) {
    h.Hin = cp.H; h.Win = cp.W; h.CGin = cp.CIG;
    h.Hout = cp.Ho; h.Wout = cp.Wo; h.NC = cp.Cout;
    h.padh = cp.pad; h.padw = cp.pad;
  } else if (!qd) {
    if (cp.pad > cp.Kh - 1 || cp.pad > cp.Kw - 1) return false;
    h.Hin = cp.Ho; h.Win = cp.Wo; h.CGin = cp.COG;
    h.Hout = cp.H; h.Wout = cp.W; h.NC = cp.Cin;
    h.padh = cp.Kh - 1 - cp.pad; h.padw = cp.Kw - 1 - cp.pad;
  } else {
    // dX[2i + a] = sum over taps kh with (a + pad - kh) even of
    // W[kh] dY[i + (a + pad - kh) / 2]: per output phase a stride-1
    // correlation over dY; the dY rows read span the offsets dmin..dmax
    // a 1-tap dimension leaves output phases no tap reaches: three quarters
    // of the tile would be zeros (the generic kernel is faster there)
    if (cp.Kh * cp.Kw > 9 || cp.Kh < 2 || cp.Kw < 2) return false;
    auto span = [&](int K, int &dmin, int &dmax) {
      dmin = 1 << 20; dmax = -(1 << 20);
      for (int k = 0; k < K; ++k) {
        const int a = ((k - cp.pad) % 2 + 2) % 2, d = (a + cp.pad - k) / 2;
        dmin = std::min(dmin, d); dmax = std::max(dmax, d);
      }
    };
    int dminh, dmaxh, dminw, dmaxw;
    span(cp.Kh, dminh, dmaxh);
    span(cp.Kw, dminw, dmaxw);
    h.QD = 1; h.qpad = cp.pad;
    // taps grouped by output phase f = 2 a + b
    int n = 0;
    for (int f = 0; f < 4; ++f) {
      h.qbeg[f] = (uint8_t)n;
      for (int t = 0; t < cp.Kh * cp.Kw; ++t) {
        const int kh = t / cp.Kw, kw = t % cp.Kw;
        const int a = ((kh - cp.pad) % 2 + 2) % 2, b = ((kw - cp.pad) % 2 + 2) % 2;
        if (2 * a + b == f) h.qorder[n++] = (uint8_t)t;
      }
    }
    h.qbeg[4] = (uint8_t)n;
    h.Hin = cp.Ho; h.Win = cp.Wo; h.CGin = cp.COG;
    h.Hout = (cp.H + 1) / 2; h.Wout = (cp.W + 1) / 2; h.NC = cp.Cin;
    h.padh = -dminh; h.padw = -dminw;
    h.HKh = dmaxh - dminh + 1; h.HKw = dmaxw - dminw + 1;
  }
  h.NPHS = qd ? 4 : 1;
  h.outH = qd ? cp.H : h.Hout;
  h.outW = qd ? cp.W : h.Wout;
  h.NCG = h.NC / 8;
  if (h.CGin % CGC) return false;
  h.nchunks = h.CGin / CGC;
  if (!qd) { h.HKh = h.Kh; h.HKw = h.Kw; }
  // positions x batch groups = 16 row groups (M = 128); least padding waste
  int best = -1;
  double best_waste = 1e30;
  for (int P = 16; P >= 1; P >>= 1) {
    const int G = 16 / P;
    if (G > h.NG || h.NG % G) continue;
    const double waste = (double)((h.Wout + P - 1) / P * P) / h.Wout;
    if (waste < best_waste - 1e-9) {
      best_waste = waste;
      best = P;
    }
  }
  if (best < 0) return false;
  h.P = best;
  h.G = 16 / best;
  const int bba = block_bytes(cp.a.fmt), bbb = block_bytes(cp.b.fmt);
  // Tile choice: output channels per tile BN and output rows per tile R, by
  // a small cost model: rounds of tiles over the SMs x time per tile.  In
  // isolation a 128 x BN x 16 MMA costs max(BN / 2, 40) cycles (narrow N runs
  // below the peak rate; N = 64 was measured at 48); a tile pays a fixed
  // pipeline fill / epilogue overhead of about two chunks.
  const int taps = h.Kh * h.Kw;
  const int bn_max = std::min(256, (h.NC + 15) / 16 * 16);
  double best_cost = 1e300;
  HaloConv best_h = h;
  bool found = false;
  // narrower than 128 columns only when the layer itself is (N < 128 MMAs run
  // below the peak rate and duplicate the halo decode across column tiles)
  const int bn_min = std::min(bn_max, 128);
  for (int BN = bn_max; BN >= bn_min; BN = BN > bn_min ? std::max(bn_min, BN / 2 / 16 * 16) : 0) {
    for (int R = 4; R >= 1; --R) {
      HaloConv c = h;
      c.BN = BN;
      c.NB = BN / 8;
      c.acc_cols = pow2_at_least32(BN);
      // accumulator ring of NS slots (all of the TMEM): rows of successive
      // tiles take successive slots, so the NS - R slots beyond a tile's own
      // let the next tile's MMAs start while the epilogue drains this one
      c.NS = std::min(MAX_R, 512 / c.acc_cols);   // a power of two
      c.ns_log2 = 0;
      while ((1 << c.ns_log2) < c.NS) ++c.ns_log2;
      c.RT = R * h.NPHS;
      if (R > h.Hout || c.RT > c.NS) continue;
      if (R > 1 && h.Kh < h.S) continue;   // the halo rows between output rows would go unused
      c.R = R;
      const size_t sm = halo_smem(c, bba, bbb);
      if (!sm) continue;
      c.smem = sm;
      const int64_t tiles = (int64_t)(h.NG / h.G) * ((h.Wout + h.P - 1) / h.P) * ((h.Hout + R - 1) / R) *
                            ((h.NC + BN - 1) / BN);
      // per chunk the MMAs and the decode of its halo + weight blocks
      // overlap; measured in this kernel (8 decode warps): ~2x the isolated
      // MMA cost with both issuers busy, ~1.6x that per MMA for one issuer
      // on its own (a tile's accumulators are split between the two issuers,
      // so one accumulator leaves one of them idle and three give one of
      // them two), and ~7.7 cycles per decoded block
      const double mma = 2.0 * std::max(BN / 2.0, BN == 64 ? 48.0 : 40.0);
      const double mmas = (double)R * taps, per_issuer = mmas * ((c.RT + 1) / 2) / c.RT;
      const double chunk_t = std::max(std::max(mmas * mma, 1.6 * per_issuer * mma),
                                      7.7 * (c.nh_blocks + c.nb_blocks));
      const double tile_t = (h.nchunks + 2.0) * chunk_t;
      const double rounds = (double)((tiles + num_sms - 1) / num_sms);
      // the epilogue of a tile (measured: ~8.5 cycles per accumulator
      // column and row with fp32 output, ~40 with the requantizing
      // epilogue) is hidden behind the next tile's MMAs as far as the ring
      // has spare slots for that tile's rows
      const double epi_t = (cp.rq.codes ? 40.0 : 8.5) * BN * c.RT;
      const int spare = c.NS - c.RT;
      const double exposed = spare >= c.RT ? 0.0 : 1.0 - (double)spare / c.RT;
      const double cost = rounds * tile_t + (rounds - 1.0) * exposed * epi_t;
      if (cost < best_cost * 0.98) {
        best_cost = cost;
        best_h = c;
        found = true;
      }
    }
    if (BN == bn_min) break;
  }
  if (!found) return false;
  h = best_h;
  // The decoded weight copy keeps the tile plan (its benefit is the weight
  // decode saved per chunk; a plan chosen for it would trade that against
  // tile overheads the cost model does not see) and frees the shared memory
  // of the packed weights.  Its box spans all taps in one dimension (at most
  // 256).
  if (cp.wdec && taps <= 256) {
    HaloConv w = h;
    w.wd = 1;
    const size_t sm = halo_smem(w, bba, bbb);
    if (sm) {
      w.smem = sm;
      h = w;
    }
  }
  h.gran_h = pow2_part(h.G * h.CGin);
  h.gran_w = h.op == OP_FWD ? pow2_part(h.CIG * std::gcd(h.COG, h.NB)) : pow2_part(std::gcd(h.CIG, h.NB));
  h.tiles_g = h.NG / h.G;
  h.tiles_w = (h.Wout + h.P - 1) / h.P;
  h.tiles_h = (h.Hout + h.R - 1) / h.R;
  h.tiles_n = (h.NC + h.BN - 1) / h.BN;
  const int64_t nt = (int64_t)h.tiles_g * h.tiles_w * h.tiles_h * h.tiles_n;
  if (nt <= 0 || nt > INT32_MAX) return false;
  h.num_tiles = (int)nt;
  return true;
}


cudaError_t halo_launch(const ConvParams &cp, HaloConv &h, int num_sms, cudaStream_t st) {
  const int bba = block_bytes(cp.a.fmt), bbb = block_bytes(cp.b.fmt);
  h.w_scales = cp.b.scales;
  h.in_scales = cp.a.scales;
  h.sa = cp.a.s_t;
  h.sb = cp.b.s_t;
  h.pre_mult = cp.pre_mult;
  h.out = cp.out;
  h.rq = cp.rq;
  h.status = cp.status;
  h.inject = cp.inject;
  // input codes [Hin][Win][NG][CGin * BBA] as 8-byte units; box: one chunk's
  // channel groups x G batch groups x WP positions x RH rows
  CUtensorMap ma, mb;
  if (h.S == 1) {
    const uint64_t d[4] = {(uint64_t)h.CGin * bba / 8, (uint64_t)h.NG, (uint64_t)h.Win, (uint64_t)h.Hin};
    const uint32_t bx[4] = {(uint32_t)(CGC * bba / 8), (uint32_t)h.G, (uint32_t)h.WP, (uint32_t)h.RH};
    if (!make_tensor_map(&ma, cp.a.codes, 8, 4, d, bx)) return cudaErrorInvalidValue;
  } else {
    // stride 2: the same codes as [Hin][Win / 2][2 (column parity)][NG][..];
    // a box holds one column phase
    const uint64_t pos = (uint64_t)h.NG * h.CGin * bba;
    const uint64_t d[5] = {(uint64_t)h.CGin * bba / 8, (uint64_t)h.NG, 2, (uint64_t)h.Win / 2, (uint64_t)h.Hin};
    const uint64_t gs[4] = {(uint64_t)h.CGin * bba, pos, 2 * pos, (uint64_t)h.Win * pos};
    const uint32_t bx[5] = {(uint32_t)(CGC * bba / 8), (uint32_t)h.G, 1u, (uint32_t)h.WP, (uint32_t)h.RH};
    if (!make_tensor_map_strided(&ma, cp.a.codes, 8, 5, d, gs, bx)) return cudaErrorInvalidValue;
  }
  if (h.wd) {
    // decoded weights [taps][COG][CIG][128 bytes] as 8-byte units; box: a
    // chunk's CGC input-channel groups x the tile's NB output-channel groups
    // (fwd), or the tile's NB input-channel groups x CGC output-channel
    // groups (dgrad), all taps -- the order the decode warps would write
    const uint64_t d[4] = {16, (uint64_t)h.CIG, (uint64_t)h.COG, (uint64_t)(h.Kh * h.Kw)};
    const uint64_t gs[3] = {128, (uint64_t)h.CIG * 128, (uint64_t)h.COG * h.CIG * 128};
    uint32_t bx[4] = {16u, 0u, 0u, (uint32_t)(h.Kh * h.Kw)};
    bx[1] = (uint32_t)(cp.op == OP_FWD ? CGC : h.NB);
    bx[2] = (uint32_t)(cp.op == OP_FWD ? h.NB : CGC);
    if (!make_tensor_map_strided(&mb, cp.wdec, 8, 4, d, gs, bx)) return cudaErrorInvalidValue;
  } else {
    // weights [taps][COG][CIG * BBB]
    const uint64_t d[3] = {(uint64_t)h.CIG * bbb / 8, (uint64_t)h.COG, (uint64_t)(h.Kh * h.Kw)};
    uint32_t bx[3];
    if (cp.op == OP_FWD) {
      bx[0] = (uint32_t)(CGC * bbb / 8); bx[1] = (uint32_t)h.NB; bx[2] = (uint32_t)(h.Kh * h.Kw);
    } else {
      bx[0] = (uint32_t)(h.NB * bbb / 8); bx[1] = (uint32_t)CGC; bx[2] = (uint32_t)(h.Kh * h.Kw);
    }
    if (!make_tensor_map(&mb, cp.b.codes, 8, 3, d, bx)) return cudaErrorInvalidValue;
  }
  const int grid = std::min(h.num_tiles, num_sms);
  const int fr = cp.rq.codes ? cp.rq.fmt : 0;
  if (cp.op == OP_FWD)
    return fr == 0 || fr == 4 ? halo_dispatch_fwd_04(cp.a.fmt, cp.b.fmt, fr, ma, mb, h, grid, st)
                              : halo_dispatch_fwd_68(cp.a.fmt, cp.b.fmt, fr, ma, mb, h, grid, st);
  return fr == 0 || fr == 4 ? halo_dispatch_dgrad_04(cp.a.fmt, cp.b.fmt, fr, ma, mb, h, grid, st)
                            : halo_dispatch_dgrad_68(cp.a.fmt, cp.b.fmt, fr, ma, mb, h, grid, st);
}


namespace {

size_t wgrad_smem(HaloWgrad &h, int bba, int bbb) {
  h.WP = h.S == 1 ? h.P + h.Kw - 1 : h.P + (h.Kw - 1) / 2;
  h.NPH = (h.S == 2 && h.Kw > 1) ? 2 : 1;
  h.PHP = h.WP;
  if (h.NPH > 1)   // each phase's packed box must start 128-byte aligned
    while ((h.PHP * h.G * h.CB * bbb) % 128) ++h.PHP;
  h.na_blocks = h.KG * 16;
  h.nb_blocks = h.NPH * h.PHP * h.G * h.CB;
  h.dec_b_off = (uint32_t)h.na_blocks * 128;
  h.dec_stage = (uint32_t)(h.na_blocks + h.nb_blocks) * 128;
  h.pk_b_off = (uint32_t)((h.na_blocks * bba + 127) / 128 * 128);
  h.pk_sc_off = (uint32_t)((h.pk_b_off + h.nb_blocks * bbb + 127) / 128 * 128);
  // bytes the boxes deliver per chunk (the phase padding is not written)
  h.pk_bytes = (uint32_t)(h.na_blocks * bba + h.NPH * h.WP * h.G * h.CB * bbb);
  h.pk_stage = (uint32_t)((h.pk_sc_off + h.na_blocks + h.nb_blocks + 127) / 128 * 128);
  const size_t fixed = 1024 + (size_t)DSTAGES * h.dec_stage + sizeof(WgCtl) + 128;
  if (fixed + 2 * (size_t)h.pk_stage > SMEM_LIMIT) return 0;
  h.PS = (int)std::min<size_t>(MAX_PS, (SMEM_LIMIT - fixed) / h.pk_stage);
  h.off_dec = 0;
  h.off_pk = DSTAGES * h.dec_stage;
  h.off_ctl = h.off_pk + h.PS * h.pk_stage;
  return 1024 + (size_t)h.off_ctl + sizeof(WgCtl);
}

constexpr int WG_TARGET_CTAS = 148;   // split-K sized for one wave on a 148-SM B300

}  // namespace

bool halo_wgrad_plan(const ConvParams &cp, HaloWgrad &h, int max_splits) {
  std::memset(&h, 0, sizeof(h));
  if (cp.op != OP_WGRAD) return false;
  // stride 2 reads X through a [H][W/2][2] view
  if (cp.stride != 1 && !(cp.stride == 2 && cp.W % 2 == 0)) return false;
  h.S = cp.stride;
  h.N = cp.N; h.NG = cp.NG; h.H = cp.H; h.W = cp.W; h.Ho = cp.Ho; h.Wo = cp.Wo;
  h.Cin = cp.Cin; h.Cout = cp.Cout; h.CIG = cp.CIG; h.COG = cp.COG;
  h.Kh = cp.Kh; h.Kw = cp.Kw; h.pad = cp.pad;
  h.ncols = cp.Kh * cp.Kw * cp.Cin;
  if (h.Kw > 16 || h.Kh > 64) return false;
  // chunk: P positions x G batch groups, 16 k-groups, least padding waste
  int best = -1;
  double best_waste = 1e30;
  for (int P = 16; P >= 1; P >>= 1) {
    const int G = 16 / P;
    if (G > h.NG || h.NG % G) continue;
    const double waste = (double)((h.Wo + P - 1) / P * P) / h.Wo;
    if (waste < best_waste - 1e-9) {
      best_waste = waste;
      best = P;
    }
  }
  if (best < 0) return false;
  h.P = best;
  h.G = 16 / best;
  h.KG = 16;   // the MMA issue loop is unrolled for K = 128 per chunk
  const int bba = block_bytes(cp.a.fmt), bbb = block_bytes(cp.b.fmt);
  h.BNc = std::min(128, (h.Cin + 15) / 16 * 16);
  for (;;) {
    h.CB = (h.BNc + 7) / 8;
    h.acc_cols = pow2_at_least32(h.BNc);
    const bool fits_tmem = h.Kw * h.acc_cols <= 512;
    if (fits_tmem && (h.smem = wgrad_smem(h, bba, bbb)) != 0) break;
    if (h.BNc <= 16) return false;
    h.BNc = std::max(16, h.BNc / 2 / 16 * 16);
  }
  if (h.BNc % 16) return false;
  h.gran_a = pow2_part(std::gcd(h.COG, 16));
  h.gran_b = pow2_part(std::gcd(h.CIG, h.CB));
  h.m_tiles = (h.Cout + 127) / 128;
  h.c_tiles = (h.Cin + h.BNc - 1) / h.BNc;
  h.tiles_w = (h.Wo + h.P - 1) / h.P;
  h.tiles_g = h.NG / h.G;
  const int64_t q = (int64_t)h.Ho * h.tiles_w * h.tiles_g;
  if (q <= 0 || q > INT32_MAX) return false;
  h.total_chunks = (int)q;
  const int groups = h.m_tiles * h.c_tiles * h.Kh;
  int s = std::max(1, WG_TARGET_CTAS / groups);
  s = std::min(s, h.total_chunks);
  if (max_splits > 0) s = std::min(s, max_splits);
  h.chunks_per_split = (h.total_chunks + s - 1) / s;
  h.splits = (h.total_chunks + h.chunks_per_split - 1) / h.chunks_per_split;   // every split non-empty
  const int64_t nt = (int64_t)groups * h.splits;
  if (nt > INT32_MAX) return false;
  h.num_tiles = (int)nt;
  return true;
}

cudaError_t halo_wgrad_launch(const ConvParams &cp, HaloWgrad &h, int num_sms, cudaStream_t st) {
  const int bba = block_bytes(cp.a.fmt), bbb = block_bytes(cp.b.fmt);
  h.a_scales = cp.a.scales;
  h.b_scales = cp.b.scales;
  h.out = cp.out;
  h.status = cp.status;
  CUtensorMap ma, mb;
  {
    // dY codes [Ho][Wo][NG][COG * BBA]; box: 16 channel groups x G x P x 1 row
    const uint64_t d[4] = {(uint64_t)h.COG * bba / 8, (uint64_t)h.NG, (uint64_t)h.Wo, (uint64_t)h.Ho};
    const uint32_t bx[4] = {(uint32_t)(16 * bba / 8), (uint32_t)h.G, (uint32_t)h.P, 1u};
    if (!make_tensor_map(&ma, cp.a.codes, 8, 4, d, bx)) return cudaErrorInvalidValue;
  }
  if (h.S == 1) {
    // X codes [H][W][NG][CIG * BBB]; box: CB channel groups x G x WP x 1 row
    const uint64_t d[4] = {(uint64_t)h.CIG * bbb / 8, (uint64_t)h.NG, (uint64_t)h.W, (uint64_t)h.H};
    const uint32_t bx[4] = {(uint32_t)(h.CB * bbb / 8), (uint32_t)h.G, (uint32_t)h.WP, 1u};
    if (!make_tensor_map(&mb, cp.b.codes, 8, 4, d, bx)) return cudaErrorInvalidValue;
  } else {
    // stride 2: X as [H][W / 2][2 (column parity)][NG][..]; a box holds one
    // column phase of one row
    const uint64_t pos = (uint64_t)h.NG * h.CIG * bbb;
    const uint64_t d[5] = {(uint64_t)h.CIG * bbb / 8, (uint64_t)h.NG, 2, (uint64_t)h.W / 2, (uint64_t)h.H};
    const uint64_t gs[4] = {(uint64_t)h.CIG * bbb, pos, 2 * pos, (uint64_t)h.W * pos};
    const uint32_t bx[5] = {(uint32_t)(h.CB * bbb / 8), (uint32_t)h.G, 1u, (uint32_t)h.WP, 1u};
    if (!make_tensor_map_strided(&mb, cp.b.codes, 8, 5, d, gs, bx)) return cudaErrorInvalidValue;
  }
  const int grid = std::min(h.num_tiles, num_sms);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h.smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, WG_THREADS, h.smem, st>>>(ma, mb, h);
    return cudaGetLastError();
  };
  const int fa = cp.a.fmt, fb = cp.b.fmt;
  if (fa == 4) {
    if (fb == 4) return go(halo_wgrad_kernel<4, 4>);
    if (fb == 6) return go(halo_wgrad_kernel<4, 6>);
    return go(halo_wgrad_kernel<4, 8>);
  }
  if (fa == 6) {
    if (fb == 4) return go(halo_wgrad_kernel<6, 4>);
    if (fb == 6) return go(halo_wgrad_kernel<6, 6>);
    return go(halo_wgrad_kernel<6, 8>);
  }
  if (fb == 4) return go(halo_wgrad_kernel<8, 4>);
  if (fb == 6) return go(halo_wgrad_kernel<8, 6>);
  return go(halo_wgrad_kernel<8, 8>);
}

}  // namespace mq
