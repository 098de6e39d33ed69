// tm_kernels.h -- parameter blocks and host launchers of the libtm kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100.cuh"

namespace tmk {

// ----------------------------------------------------------------- bf16 tensor-core path (c_z = c_h = 128)
constexpr int kC = 128;  // channels of z and of the hidden a/b/x on the tensor-core path

// Projection: a, b = sigmoid(W_g* zh) * (W_* zh) * m_i m_j, channel-major bf16.
struct ProjectParams {
  __nv_bfloat16* a;       // [128][N][ld]
  __nv_bfloat16* b;       // [128][N][ld]
  const float* mask;      // [N] token mask of the rows i, or nullptr (ones)
  const float* mask_col;  // [N] token mask of the columns j, or nullptr (ones); the whole grid's is mask
  const float* consts;    // [2 halves][512]: rowsum[256] then bias[256] of the folded LayerNorm
  float2* zstat;          // [N][N] (rstd, -rstd mu) of LayerNorm_in per pair, written by the a-half CTA
                          // for the finish kernel; nullptr: not written
  int N, ld;
  int tiles_per_row;      // ceil(N / 128)
  long long total_tiles;  // N * tiles_per_row
  int out_f16;            // 1: a, b stored as fp16 of their bf16 values times out_scale[half] (backward)
  float out_scale[2];
  Watch w;
};

// Storage of the contraction's output x between the contraction and the finish kernels: float32,
// or fp16 scaled by one power of two 2^e.
enum XFormat : int { X_F32 = 0, X_F16 = 1 };

// The fp16 storage of x scales every value by 2^e, chosen on the host from a bound on |x| that the
// weights alone fix (tm_api.cu, x16_exponent).

// Contraction of one output block: x[c][i-i0][j-j0] over k in [0, N).
struct ContractParams {
  void* x;                // block buffer [128][bi][ldx], float32 or fp16 (x_f16)
  long long ldx;          // row stride (elements)
  long long chan_stride;  // channel stride (elements)
  int N;                  // contraction length
  int i0, j0, bi, bj;     // block origin and extents
  int i_base, j_base;     // tile grid origin: i0, j0 rounded down to a multiple of 8, so that
                          // every TMA box starts on a 16-byte boundary along its inner axis
  int tiles_i, tiles_j;   // tiles covering [i_base, i0 + bi) x [j_base, j0 + bj)
  long long total_tiles;  // 128 * tiles_i * tiles_j
  int last_n;             // MMA N of the last tile column: the columns it still has to cover, rounded up to 16
  int x_f16;              // 1: x is stored fp16, scaled by 2^x_exp
  int x_exp;
  int ab_f16;             // 1: a and b are fp16 (the backward pass's operands), else bf16
  int accumulate;         // 1: float32 x += the product (TMA reduce-add; needs tma_store), else x = it
  int tma_store;          // 1: x leaves through TMA stores (needs i0, j0 multiples of 8); 0: direct stores
  Watch w;
};

// Output epilogue of one block: out = sigmoid(g) * (W_o LayerNorm(x)).
struct FinishParams {
  // rowsum of W_g' (hi+lo), bias W_g beta_in, bias W_o beta_out, rowsum of W_o' (times inv_scale_o);
  // all halved for the tanh form. First and 16-byte aligned: the epilogue reads them two at a time as
  // 8-byte constant-bank operands.
  alignas(16) float cst[4 * kC];
  int x_exp;              // fp16 x is stored times 2^x_exp
  int residual;           // 1: out += update (out holds z: a residual connection), else out = update
  const float2* zstat;    // [N][N] (rstd, -rstd mu) of LayerNorm_in per pair (fp16-x kernel)
  float inv_scale_o;      // W_o is stored scaled by a power of two; this undoes it
  int N;
  int i0, j0, bi, bj;
  int tiles_j;            // ceil(bj / 128)
  long long total_tiles;  // bi * tiles_j
  Watch w;
};

cudaError_t launch_project_bf16(const CUtensorMap& zmap, const CUtensorMap& wmap, const CUtensorMap& amap,
                                const CUtensorMap& bmap, const ProjectParams& p, int num_sms, cudaStream_t s);
// The contraction's operand forms: outgoing x_ij = sum_k a_ik b_jk, incoming x_ij = sum_k a_ki b_kj, and
// mixed x_ij = sum_k a_ik b_kj (float32 x only).
enum ContractMode : int { CONTRACT_OUT = 0, CONTRACT_IN = 1, CONTRACT_MIXED = 2 };
cudaError_t launch_contract_bf16(int mode, const CUtensorMap& amap, const CUtensorMap& bmap,
                                 const CUtensorMap& xmap, const ContractParams& p, int num_sms, cudaStream_t s);
// x16 selects the fp16 x tile (kBoxFinishX16, double-buffered) instead of the float32 one.
cudaError_t launch_finish_bf16(bool x16, const CUtensorMap& xmap, const CUtensorMap& zmap,
                               const CUtensorMap& womap, const CUtensorMap& wgmap, const CUtensorMap& omap,
                               const FinishParams& p, int num_sms, cudaStream_t s);

// Tile sizes.
constexpr int kProjTileJ = 128;     // pairs per projection tile
constexpr int kContractBM = 256;    // output rows per contraction tile (a CTA pair, 128 rows each)
constexpr int kContractBN = 256;    // output columns per contraction tile (128 B rows staged by each CTA)
constexpr int kContractBK = 64;     // k per pipeline stage
constexpr int kFinishTileJ = 128;   // pairs per finish tile

// Box shape (elements, innermost first) and element size of every tensor map. The host encodes the
// maps from these and each kernel checks at compile time that a box fills exactly the shared-memory
// slot it is copied into (a larger box would write past the slot).
struct Box {
  uint32_t d0, d1, d2, esz;
  __host__ __device__ constexpr uint32_t bytes() const { return d0 * d1 * d2 * esz; }
};
constexpr Box kBoxProjZ{64, (uint32_t)kProjTileJ, 1, 2};              // z tile, one 64-channel half
constexpr Box kBoxProjW{64, 128, 1, 2};                               // one K-half of a 128 x 128 weight
constexpr Box kBoxProjOut{32, 1, 32, 2};                              // a or b store: 32 pairs x 32 channels
constexpr Box kBoxContractOutA{(uint32_t)kContractBK, (uint32_t)kContractBM / 2, 1, 2};   // one CTA's A rows
constexpr Box kBoxContractOutB{(uint32_t)kContractBK, (uint32_t)kContractBN / 2, 1, 2};   // one CTA's B rows
constexpr Box kBoxContractIn{64, (uint32_t)kContractBK, 1, 2};        // incoming: 64-wide slab of i or j
constexpr Box kBoxContractX{32, 32, 1, 4};                            // x store sub-tile (float32)
constexpr Box kBoxContractX16{64, 32, 1, 2};                          // x store sub-tile (fp16)
constexpr Box kBoxFinishX{(uint32_t)kFinishTileJ, 1, (uint32_t)kC, 4};
constexpr Box kBoxFinishX16{64, 1, (uint32_t)kC, 2};                  // fp16 x: 64 pairs x 128 channels
constexpr Box kBoxFinishZ{64, (uint32_t)kFinishTileJ, 1, 2};
constexpr Box kBoxFinishW{64, (uint32_t)kC, 1, 2};                    // W_o (fp16) and W_g (bf16) halves
constexpr Box kBoxFinishOut{64, 32, 1, 2};                            // out store: 32 pairs x 64 channels

// ----------------------------------------------------------------- float32 CUDA-core path (any c <= 256)
struct F32Weights {
  const float *ln_in_g, *ln_in_b, *w_a, *w_ga, *w_b, *w_gb, *w_g, *ln_out_g, *ln_out_b, *w_o;
  int c_z, c_h;
};

cudaError_t launch_project_f32(const float* z, const float* mask, const F32Weights& w, float* a, float* b,
                               int N, int ld, cudaStream_t s);
cudaError_t launch_contract_f32(bool incoming, const float* a, const float* b, int N, int ld, int c_h, int i0,
                                int j0, int bi, int bj, float* x, long long ldx, long long chan_stride,
                                cudaStream_t s);
cudaError_t launch_finish_f32(const float* x, long long ldx, long long chan_stride, const float* z,
                              const F32Weights& w, int N, int i0, int j0, int bi, int bj, float* out,
                              bool residual, cudaStream_t s);

// Backward pass (k_f32_backward.cu). Per-pair vectors are channel-major [c][N*N] (pair p = i*N + j);
// the gradient planes dX, dXT, dA, dB are [c_h][N][ld].
struct BwdF32Vectors {
  float *dX, *dXT;                  // dL/dx and its per-channel transpose (output backward)
  const float *dA, *dB;             // dL/da, dL/db (contraction gradients)
  int ld;
  float* dzh;                       // [c_z][P] dL/dzh: the gate's term, then the projections' terms
  float *zh, *xh, *dy, *dgg;        // [c_z], [c_h], [c_z], [c_z] x [P]
  float *q_out_n, *q_out;           // [c_h][P] dxh * n_x and dxh
  float *dpa, *dga, *dpb, *dgb;     // [c_h][P]
  float *q_in_n, *q_in;             // [c_z][P] dzh * n_z and dzh
};
constexpr int kOuterSumMaxSplits = 512;
cudaError_t launch_bwd_output_f32(const float* x, long long ldx, const float* z, const float* dout,
                                  const F32Weights& w, int N, const BwdF32Vectors& v, cudaStream_t s);
cudaError_t launch_bwd_project_f32(const float* z, const float* mask, const F32Weights& w, int N,
                                   const BwdF32Vectors& v, float* dz, cudaStream_t s);
// out[o][k] = sum_p U[o][p] V[k][p] (V == nullptr: K = 1, V = 1) through outer_sum_splits(P) fixed-order
// partial sums in part [splits][O][K].
int outer_sum_splits(long long P);
cudaError_t launch_outer_sum_f32(const float* U, const float* V, int O, int K, long long P, float* part,
                                 float* out, cudaStream_t s);

// Backward pass, bf16 tensor-core path (k_backward.cu). Pairs are taken in tiles of 128 consecutive
// entries of the flattened grid (p = i * N + j); per-pair vectors are channel-major [128][N * N]. Every
// tensor-core operand is fp16, stored times a power of two; the u_* factors undo, in each product's
// epilogue, the scales its operands carry (the host's part; a part set by a recorded maximum, amax, is
// computed on the device).
// Output backward over one block of the pair grid: pairs (i0 + il, j0 + jl), il < bi, jl < bj (the whole
// grid: 0, 0, N, N), with x the contraction's block [128][bi][ldx].
struct BwdOutParams {
  const __nv_bfloat16* z;         // [N][N][128]
  const float2* zstat;            // [N][N] (rstd, -rstd mu) of LayerNorm_in (projection kernel)
  const float* x;                 // [128][bi][ldx] float32: the contraction's x times 1 / x_unscale
  long long ldx, xplane;          // row and channel strides of x
  float x_unscale;
  const __nv_bfloat16* dout;      // [N][N][128]
  unsigned* amax;                 // [0] largest |dout| (read); [1] the bound on |dX| that fixes dX's fp16
                                  // scale (written); [2] largest |dX| (merged in); float bits
  float dx_bound;                 // |dX| <= dx_bound * largest |dout|
  float y_bound4;                 // bound on |W_o xh| / 4 (dgg's scale)
  float sz, sx;                   // zh, xh are stored times sz, sx
  float u_gg, u_y;                // gg = MMA * u_gg, y = MMA * u_y
  float u_dxh, u_dzh, u_wg, u_wo; // dxh, dzh_g, dW_g, dW_o: host parts of the unscale
  __half* dx16;                   // [128][N][ldd] fp16 dL/dx times its scale, or nullptr (not written)
  long long ldd, dxplane;
  float* dzh;                     // [128][dzh_P]: the gate's term of dL/dzh of pair p at p - dzh_off, or
  long long dzh_P, dzh_off;       // nullptr (not written)
  float* part_w;                  // [grid][2][128][128] per-CTA sums of dW_g, dW_o (added to), or nullptr
  float* part_ln;                 // [grid][256] per-CTA sums of d(gamma_out), d(beta_out) (added to)
  const __half *w_g, *w_o;        // fp16 weight images (times powers of two) in the swizzled tile layout
  const float* ln;                // gamma_in, beta_in, gamma_out, beta_out (float32, 4 x 128)
  int N;
  int i0, j0, bi, bj;
  long long tiles;                // ceil(bi bj / 128)
  Watch w;
};
// Projection backward over the pairs [p0, p0 + P) of the flattened grid (whole rows: p0 = i_off N).
struct BwdProjParams {
  const __nv_bfloat16* z;
  const float2* zstat;
  const float* mask;              // [N] or nullptr
  const float* dV;                // [128][rows][ldv] float32, rows i_off.. : dL/da or dL/db times (dX's
                                  // scale x partner's)
  long long ldv, vplane;
  const unsigned* amax;           // [1] the bound on |dX|, which fixes dX's scale; [2] largest |dX| (bits)
  float sz;                       // zh is stored times sz
  float u_pv, u_pg;               // pv = MMA * u_pv, pg = MMA * u_pg
  float q_raw, q2f;               // |dV| <= q_raw x (largest fp16 dX); |dpg| / |dpv| <= q2f
  float u_dzh_v, u_dzh_g, u_wv, u_wgt;   // host parts of the unscales of the W^T products and dW
  float* dzh;                     // [128][dzh_P], pair p at p - dzh_off, accumulated
  long long dzh_P, dzh_off;
  __nv_bfloat16* dz;              // [N][N][128] (final pass)
  int final_pass;                 // 1: add this side's term, then LayerNorm_in backward into dz
  float* part_w;                  // [grid][2][128][128] per-CTA sums of dW_v, dW_gt (added to)
  float* part_ln;                 // [grid][256] per-CTA sums of d(gamma_in), d(beta_in) (final pass, added to)
  const __half *w_v, *w_gt;
  const float* ln;                // gamma_in, beta_in
  int N;
  int i_off;
  long long p0, P, tiles;
  Watch w;
};
int bwd_grid(long long tiles, int num_sms);
cudaError_t launch_bwd_output_bf16(const BwdOutParams& p, int grid, cudaStream_t s);
cudaError_t launch_bwd_project_bf16(const BwdProjParams& p, int grid, cudaStream_t s);
// *out = max(*out, bits of the largest |v|) over n bf16 values
cudaError_t launch_absmax_bf16(const __nv_bfloat16* v, long long n, unsigned* out, int num_sms, cudaStream_t s);
// out[e] = sum over q < S of part[q * stride + e], e < E, in order q = 0, 1, ...
cudaError_t launch_sum_parts(const float* part, int S, long long E, long long stride, float* out, cudaStream_t s);
// The same for up to 10 jobs in one launch (a job whose out is nullptr is skipped).
struct SumJobs {
  const float* part[10];
  float* out[10];
  long long E[10], stride[10];
  int n;
};
cudaError_t launch_sum_parts_multi(const SumJobs& j, int S, cudaStream_t s);

// Triangle attention, tensor-core path (k_attention.cu): bf16 z and out, fp16 intermediates, c_z = 128,
// 4 heads of 32. The grid may be
// the transposed one (ending node): pair (i, j) then reads z at (j, i) and writes out at (j, i).
struct TaProjectParams {
  const __nv_bfloat16* z;           // [N][N][128]
  const float* mask;                // [N] or nullptr: keys j with mask 0 get a bias of -inf
  int transpose;
  const float* ln;                  // gamma, beta (float32, 2 x 128), both times 2^sz (zh is stored scaled)
  const float* w_b;                 // [4][128] float32
  const __half *w_q, *w_k, *w_v, *w_g;   // fp16 tile images, each scaled by a power of two
  float wscale[4];                  // per product: undoes the image's and zh's scales; q's also carries
                                    // log2(e)/sqrt(c), v's the power of two v is stored times
  float bscale;                     // log2(e) 2^-sz: the bias of the scaled zh in base-2 logit units
  __half *q, *k, *g;                // [N][N][128] pair-major
  __half* vt;                       // [N][128][ldv]: row i, (head, channel), key
  __half* b;                        // [4][N][ldb]: head, j, k (times log2(e); -inf at masked keys)
  long long ldv, ldb;
  int N;
  long long P, tiles;
  Watch w;
};
struct TaAttendParams {
  const float* mask;                // [N] or nullptr
  const __half* g;                  // [N][N][128]
  __half* o;                        // [N][N][128]: gated attention output of every head
  int N, jpairs;                    // jpairs: pairs of 128-query tiles per row, ceil(ceil(N / 128) / 2)
  Watch w;
};
struct TaOutParams {
  const __half* o;
  const __half* w_o;                // fp16 tile image of W_o [128][128], scaled by a power of two
  float oscale;                     // undoes that scale and the scale of the stored o (that of v)
  __nv_bfloat16* out;               // [N][N][128]
  int transpose;
  int N;
  long long P, tiles;
  Watch w;
};
cudaError_t launch_ta_project(const TaProjectParams& p, int grid, cudaStream_t s);
cudaError_t launch_ta_attend(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const CUtensorMap& bmap, const TaAttendParams& p, cudaStream_t s);
cudaError_t launch_ta_out(const TaOutParams& p, int grid, cudaStream_t s);
// Box shapes of the attention kernel's tensor maps (elements innermost first, 128-byte swizzle).
constexpr Box kBoxTaQK{64, 128, 1, 2};     // 64 channels (a head pair) x 128 positions of one row
constexpr Box kBoxTaV{64, 32, 1, 2};       // 64 keys x 32 channels of one head of one row
constexpr Box kBoxTaK{64, 64, 1, 2};      // 64 channels (a head pair) x 64 keys of one row
constexpr Box kBoxTaBias{64, 128, 1, 2};   // 64 keys x 128 queries of one head

// The dynamic shared-memory limit of a kernel is a property of the kernel's instance on one device
// (cudaFuncSetAttribute acts on the current device), so the launchers raise it once per device rather
// than once per process; later launches, including those recorded into a CUDA graph, find it set.
constexpr int kMaxDevices = 64;
template <typename F>
cudaError_t once_per_device(bool (&done)[kMaxDevices], F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  e = set();
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// ----------------------------------------------------------------- diagnostics
enum : int { KID_SELFTEST = 9 };
cudaError_t launch_watchdog_selftest(const Watch& w, cudaStream_t s);
// blocks CTAs of 512 threads, each thread 8 x iters ex2.approx.ftz.f32
cudaError_t launch_probe_ex2(int blocks, int iters, cudaStream_t s);

}  // namespace tmk
