// kernels.h -- host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mq {

// bytes of one packed 8x8 block for element format fmt (4, 6 or 8 bits)
__host__ __device__ constexpr int block_bytes(int fmt) { return fmt == 4 ? 32 : fmt == 6 ? 48 : 64; }

struct QuantParams {
  int64_t d0, d1, d2, d3;          // ACT/GRAD: N, C, H, W; WEIGHT: Cout, Cin, Kh, Kw
  uint8_t *codes;
  uint8_t *scales;
  float *s_t_out;
  const uint32_t *amax_src_bits;   // statistic T_scale is built from (fp32 bits)
  uint32_t *amax_meas_bits;        // nullable: receives max |x| (atomic max of fp32 bits)
  uint32_t *status;
  int sr;                          // element codes: 0 round-to-nearest, 1 stochastic (Philox key sr_seed)
  uint64_t sr_seed;
};

enum ConvOp : int { OP_FWD = 0, OP_DGRAD = 1, OP_WGRAD = 2 };

// k-groups (8 reduction elements each) per pipeline stage of the generic
// implicit-im2col kernel (conv.cu); its weight-gradient splits are whole
// multiples of it
constexpr int CONV_KCH = 8;

struct Operand {
  const uint8_t *codes;
  const uint8_t *scales;
  const float *s_t;
  int fmt;
};

struct Requant {                   // fused requantizing epilogue of the forward conv
  uint8_t *codes;
  uint8_t *scales;
  float *s_t_out;
  const float *amax_in;
  uint32_t *amax_out_bits;         // nullable
  int fmt;
  int sr;                          // element codes: 0 round-to-nearest, 1 stochastic (Philox key sr_seed)
  uint64_t sr_seed;
};

struct ConvParams {
  int op;
  // geometry
  int N, Cin, H, W, Cout, Kh, Kw, stride, pad, Ho, Wo;
  int NG, CIG, COG;
  // operands: fwd (A = X, B = W), dgrad (A = dY, B = W), wgrad (A = dY, B = X)
  Operand a, b;
  float pre_mult;                  // undoes the operand pre-scaling of the decode
  float *out;                      // fwd: Y HWCN (nullable with rq); dgrad: dX HWCN; wgrad: partial sums
  Requant rq;                      // rq.codes == nullptr: no fused epilogue
  const void *wdec;                // fwd / dgrad: decoded weight copy (128 bytes per block, packed order)
                                   // or nullptr
  // tiling
  int BN;                          // columns per tile (multiple of 16, <= 256)
  int acc_stride;                  // TMEM columns per accumulator buffer (power of two)
  int m_tiles, n_tiles, k_splits;
  int kg_total;                    // fwd: taps*CIG; wgrad: Ho*Wo*NG
  int kg_per_split;                // wgrad
  int wg_rows;                     // wgrad: Cout rounded to 128 (partial-sum row pitch = Cout)
  int ncols;                       // wgrad: Kh*Kw*Cin
  uint32_t *status;
  int inject;                      // fault injection for the failure-detection tests (0: none)
};

// Fault injections (test support): INJECT_WITHHOLD_ACC_RELEASE makes the
// first accumulator slot of CTA 0 of the halo forward / data-gradient kernel
// expect one release more than its epilogue warps give, so the MMA issuer's
// bounded wait to reuse that slot expires (no copy or MMA is left waiting on
// it).
constexpr int INJECT_WITHHOLD_ACC_RELEASE = 1;

// Forward / data-gradient convolution (stride 1 or 2) with per-tile halo
// reuse (conv_halo.cu).  Filled by halo_plan() from a ConvParams.
struct HaloConv {
  int op;
  int N, NG;
  int Hin, Win, CGin;            // correlation input (fwd: X; dgrad: dY) and its channel groups (K)
  int Hout, Wout, NC, NCG;       // output dims and channels (fwd: Ho, Wo, Cout; dgrad: H, W, Cin)
  int Kh, Kw, padh, padw;        // taps and padding of the correlation (dgrad: K - 1 - pad)
  int P, G, R, WP, RH;           // tile: positions, batch groups, output rows; halo width (per
                                 // column phase) / height
  int S, NPH;                    // stride; halo column phases (stride 2: even / odd input columns
                                 // staged apart, so every tap reads unit-stride halo positions)
  int PHP;                       // halo positions per phase: RH * WP, padded so that every phase's
                                 // packed box starts 128-byte aligned
  int HKh, HKw;                  // halo extent in taps (Kh, Kw except for QD)
  int QD;                        // stride-2 data gradient: a tile covers R rows x P positions of output
                                 // quads (2 x 2 dX pixels), one accumulator per (row, output phase)
  int NPHS, RT;                  // accumulator phases per row (4 with QD, else 1); accumulators per tile R NPHS
  int qpad;                      // QD: padding of the forward convolution
  uint8_t qorder[9], qbeg[5];    // QD: taps grouped by output phase; phase f owns qorder[qbeg[f] .. qbeg[f + 1])
  int outH, outW;                // output rows / columns (Hout, Wout count quads with QD)
  int NS, ns_log2;               // accumulator slots (TMEM ring, a power of two; accumulator a of tile k
                                 // uses slot (k RT + a) % NS)
  int BN, NB, acc_cols;          // output channels per tile, their groups, TMEM columns per row
  int nchunks;                   // CGin / 2
  int tiles_g, tiles_w, tiles_h, tiles_n, num_tiles;
  int PS;                        // packed ring depth
  int wd;                        // 1: the weight operand is copied decoded (ConvParams::wdec) by TMA
                                 // into the decoded stages, and the decode warps convert the halo only
  uint32_t wd_bytes;             // decoded weight bytes per chunk (nb_blocks * 128)
  const uint8_t *w_scales, *in_scales;
  int COG, CIG;                  // weight block groups: W is [Kh*Kw][COG][CIG]
  const float *sa, *sb;
  float pre_mult;
  float *out;                    // fp32 HWCN, nullable with rq
  Requant rq;
  uint32_t *status;
  int inject;                    // fault injection (INJECT_*; 0: none)
  // shared-memory carve-up (bytes from the 1 KB-aligned base)
  uint32_t off_dec, dec_stage, dec_b_off;
  uint32_t off_pk, pk_stage, pk_b_off, pk_bytes;
  uint32_t off_sc, sc_bytes, sc_stride, scw_off;   // per-tile scales: halo runs, then weight runs
  uint32_t off_ctl;
  int nh_blocks, nb_blocks;
  int gran_h, gran_w;            // cp.async granules of the scale runs
  size_t smem;
};

// Weight gradient (stride 1 or 2) with per-chunk halo reuse (conv_halo.cu).  Each
// CTA tile accumulates one kernel row (kh) x Kw taps x BNc input channels x
// 128 output channels over a range of (output row, positions, batch groups)
// chunks and writes one split-K partial.
struct HaloWgrad {
  int N, NG, H, W, Ho, Wo, Cin, Cout, CIG, COG, Kh, Kw, pad;
  int P, G, KG, WP;              // chunk: P positions x G batch groups = KG k-groups (K = 8 KG);
                                 // X halo width per column phase
  int S, NPH, PHP;               // stride; X halo column phases and positions per phase (as in HaloConv)
  int BNc, CB, acc_cols;         // input channels per tile, their groups, TMEM columns per tap
  int m_tiles, c_tiles, splits, chunks_per_split, total_chunks;
  int tiles_w, tiles_g;
  int num_tiles;
  int PS;
  const uint8_t *a_scales, *b_scales;   // dY, X
  float *out;                    // partial sums [split][Cout][Kh * Kw * Cin]
  int ncols;
  uint32_t *status;
  uint32_t off_dec, dec_stage, dec_b_off;
  uint32_t off_pk, pk_stage, pk_b_off, pk_sc_off, pk_bytes;
  uint32_t off_ctl;
  int na_blocks, nb_blocks;
  int gran_a, gran_b;
  size_t smem;
};

bool halo_plan(const ConvParams &cp, HaloConv &h, int num_sms);
// max_splits <= 0: no limit
bool halo_wgrad_plan(const ConvParams &cp, HaloWgrad &h, int max_splits);
cudaError_t halo_wgrad_launch(const ConvParams &cp, HaloWgrad &h, int num_sms, cudaStream_t s);
cudaError_t halo_launch(const ConvParams &cp, HaloConv &h, int num_sms, cudaStream_t s);
// launches of the forward / data-gradient halo kernel for operand formats fa
// (input), fb (weights) and requantized-output format fr (0: none), split
// over translation units by fr (conv_halo_{fwd,dgrad}_{a,b}.cu)
#define MQ_HALO_DISPATCH(name)                                                                            \
  cudaError_t name(int fa, int fb, int fr, const CUtensorMap &a, const CUtensorMap &b, const HaloConv &h, \
                   int grid, cudaStream_t st);
MQ_HALO_DISPATCH(halo_dispatch_fwd_04)
MQ_HALO_DISPATCH(halo_dispatch_fwd_68)
MQ_HALO_DISPATCH(halo_dispatch_dgrad_04)
MQ_HALO_DISPATCH(halo_dispatch_dgrad_68)
#undef MQ_HALO_DISPATCH
// Tiled TMA descriptor of a row-major tensor (dims[0] innermost, elements of
// esize bytes) with box `box`, zero fill outside; `map` is a 64-byte aligned
// CUtensorMap.  False if the driver entry point or the encode fails.
bool make_tensor_map(void *map, const void *base, int esize, int rank, const uint64_t *dims, const uint32_t *box);
// The same with explicit byte strides of dims 1 .. rank-1 (multiples of 16).
bool make_tensor_map_strided(void *map, const void *base, int esize, int rank, const uint64_t *dims,
                             const uint64_t *strides, const uint32_t *box);

cudaError_t launch_amax(const void *src, int dtype, int64_t n, uint32_t *amax_bits, int num_sms, cudaStream_t s);
// the decoded weight copy: nblocks packed blocks of format fmt -> 128 bytes each
cudaError_t launch_weight_decode(const uint8_t *codes, const uint8_t *scales, int fmt, int64_t nblocks, void *out,
                                 int num_sms, cudaStream_t s);
cudaError_t launch_quantize(const void *src, int dtype, int layout, int fmt, const QuantParams &p, int num_sms,
                            cudaStream_t s);

// Fills the tiling fields of p for `num_sms` and returns the number of tiles.
int64_t conv_plan(ConvParams &p);
size_t conv_smem_bytes(const ConvParams &p);
cudaError_t launch_conv(const ConvParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_wgrad_reduce(const ConvParams &p, float *dw, cudaStream_t s);

}  // namespace mq
