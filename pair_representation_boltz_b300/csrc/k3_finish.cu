// k3_finish.cu -- output stage of the triangle multiplicative update on the
// sm_103a tensor cores, over one output block:
//
//   out_ij = sigmoid(W_g zh_ij) * W_o LayerNorm_out(x_ij),   zh = LayerNorm_in(z)
//
// x comes channel-major [128][bi][ldx] from the contraction; z and out are the
// caller's bf16 [N][N][128] pair representation (the layer(x, mask) call of
// the code-sample section of "NVIDIA BioNeMo escala modelagem biomolecular com
// context parallelism e quebra barreira de memória da GPU").
//
// Both LayerNorms are folded into the GEMMs' epilogue, the way the projection
// folds its input LayerNorm: with W' = W diag(gamma),
//   W LayerNorm(v) = rstd (W' v - mu rowsum W') + W beta,
// so the tensor cores read the stored operands as they are and only the
// per-pair mean and rstd are computed on the CUDA cores. For z that is exact
// (bf16 values); for x it costs nothing in accuracy either, because x is
// already stored at the precision the operand needs.
//
// Two kernels, one per storage of x:
//   k3_finish_x16  x fp16 scaled by 2^x_exp: the x tile is the MMA's
//                  A operand directly (M-major, 128-byte swizzle), two tiles in
//                  flight; LayerNorm is scale-free apart from its epsilon,
//                  which is scaled to match.
//   k3_finish_x32  x float32: the LayerNorm warps normalise it into an fp16
//                  K-major operand first (float32 does not enter kind::f16).
//
// Per tile of 128 pairs (one row i, 128 consecutive j of the block):
//   warp 0      TMA: x tile, z tile (two 64-channel boxes, 128-byte swizzle);
//               W_o' (fp16) and W_g' (bf16 hi + lo) once.
//   warp 1      tcgen05.mma: D[p][0..128) = x W_o'^T (kind::f16),
//               D[p][128..256) = z W_g'^T (bf16, hi and lo), two TMEM buffers.
//   warps 2..5  statistics, two lanes per pair (one per channel half): a shifted
//               one-pass sum and sum of squares per half, merged across the two
//               lanes (pairwise update of mean and sum of squares, Chan, Golub,
//               LeVeque), of x (and of z for float32 x; with fp16 x the
//               projection kernel's LayerNorm_in statistics are read instead);
//               handed to the epilogue through shared memory behind mbarriers.
//   warps 6..13 epilogue, thread = pair: two warps per TMEM lane quadrant split
//               the 128 output channels; folded LayerNorms, gate (sigmoid through
//               one tanh) and product, staged in shared memory and written by one
//               TMA store of 32 pairs x 64 channels per warp.
// The per-channel constants travel in the kernel's parameter block.
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int BM = kFinishTileJ;             // pairs per tile
constexpr int XS_BYTES = kC * BM * 4;        // x: one float32 [c][j] tile, or two fp16 tiles
constexpr int XH_BYTES = BM * kC * 2;        // 32 KB: out staging (and float32 x's x-hat operand)
constexpr int Z_BYTES = BM * kC * 2;         // 32 KB bf16, two K-chunks
constexpr int WO_BYTES = kC * kC * 2;        // 32 KB fp16
constexpr int WG_BYTES = 2 * kC * kC * 2;    // 64 KB bf16 hi + lo
constexpr int ST_BYTES = BM * 16;            // per-pair statistics, float4 (rstd_z, -rstd_z mu_z, rx, nx)
constexpr int LN_WARPS = 4, EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * (LN_WARPS + EPI_WARPS);
constexpr int TMEM_COLS = 512;

// mbarriers and flags, after the tiles
struct Bars {
  uint64_t xfull[2], xempty[2];   // x slots
  uint64_t zfull, zempty;         // z tile
  uint64_t hfull, hempty;         // x-hat operand (float32 x only)
  uint64_t tfull[2], tempty[2];   // TMEM accumulators
  uint64_t sfull[2], sempty[2];   // statistics (index 0 used)
  uint64_t wfull, fin;
  uint32_t tslot;
  int abort_flag;
};
constexpr int SMEM_BYTES = Z_BYTES + XH_BYTES + WO_BYTES + WG_BYTES + XS_BYTES + ST_BYTES + 256;
static_assert(sizeof(Bars) <= 256, "barrier block");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(kBoxFinishX.bytes() == XS_BYTES && 4 * kBoxFinishX16.bytes() == XS_BYTES, "x tiles");
static_assert(2 * kBoxFinishZ.bytes() == Z_BYTES, "z tile = two boxes");
static_assert(2 * kBoxFinishW.bytes() == WO_BYTES && 4 * kBoxFinishW.bytes() == WG_BYTES, "weight boxes");
static_assert(EPI_WARPS * kBoxFinishOut.bytes() == XH_BYTES && kBoxFinishOut.d0 * 2 == 128,
              "out staging: one 32-row box of 128-byte rows per epilogue warp");

// Shared-memory layout common to both kernels (1024-aligned swizzled tiles first).
struct Smem {
  uint8_t *zs, *xh, *wo, *wg, *xs;
  float4* st;
  Bars* bars;
  __device__ explicit Smem(uint8_t* base) {
    zs = base;
    xh = zs + Z_BYTES;
    wo = xh + XH_BYTES;
    wg = wo + WO_BYTES;             // hi chunks then lo chunks
    xs = wg + WG_BYTES;
    st = reinterpret_cast<float4*>(xs + XS_BYTES);
    bars = reinterpret_cast<Bars*>(xs + XS_BYTES + ST_BYTES);
  }
};

__device__ __forceinline__ float2 bf2f(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// Mean and rstd of 128 channels from two lanes' (mean, M2) over 64 channels each (lane l and l^16).
__device__ __forceinline__ void merge_halves(float mean_h, float m2_h, float eps, float& mean, float& rstd) {
  const float mean_o = __shfl_xor_sync(0xffffffffu, mean_h, 16);
  const float m2_o = __shfl_xor_sync(0xffffffffu, m2_h, 16);
  const float dm = mean_h - mean_o;
  mean = 0.5f * (mean_h + mean_o);
  const float var = fmaxf((m2_h + m2_o + 32.0f * dm * dm) * (1.0f / kC), 0.f);
  rstd = rsqrtf(var + eps);
}

// Statistics of z over its 128 channels for rows zr0 and zr0 + 16, this lane's K-chunk hc of the
// z tile (128-byte swizzle), each half shifted by its first value.
__device__ __forceinline__ void z_stats(const uint8_t* zs, int zr0, int hc, float (&mean)[2], float (&rstd)[2]) {
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = zr0 + 16 * rr;
    const uint8_t* zrow = zs + hc * (Z_BYTES / 2);
    uint4 raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) raw[u] = *reinterpret_cast<const uint4*>(zrow + sw128_offset(row, u));
    const float sh = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(&raw[0].x));
    const float2 nsh = make_float2(-sh, -sh);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0, q0 = a0, q1 = a0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float2 d0 = __fadd2_rn(bf2f(raw[u].x), nsh), d1 = __fadd2_rn(bf2f(raw[u].y), nsh);
      const float2 d2 = __fadd2_rn(bf2f(raw[u].z), nsh), d3 = __fadd2_rn(bf2f(raw[u].w), nsh);
      a0 = __fadd2_rn(a0, __fadd2_rn(d0, d2));
      a1 = __fadd2_rn(a1, __fadd2_rn(d1, d3));
      q0 = __ffma2_rn(d0, d0, __ffma2_rn(d2, d2, q0));
      q1 = __ffma2_rn(d1, d1, __ffma2_rn(d3, d3, q1));
    }
    const float2 as = __fadd2_rn(a0, a1), qs = __fadd2_rn(q0, q1);
    const float sd = as.x + as.y;
    merge_halves(sh + sd * (1.0f / 64), (qs.x + qs.y) - sd * sd * (1.0f / 64), 1e-5f, mean[rr], rstd[rr]);
  }
}

// Epilogue of one tile for one thread: pair row of the TMEM accumulator at `tmem_row`, output
// channels [64*H, 64*H + 64), written as bf16 into row `r` of the 128-byte-swizzled staging box
// `stg`. st = (rstd_z, -rstd_z mu_z, rx, nx): with FOLD_X the y accumulator holds W_o' x16 and
// y/2 = rx acc + nx rowsum' + bias'; otherwise it holds W_o' x-hat and y/2 = inv acc + bias'.
// H is a template parameter so the constant-bank offsets are immediates.
template <int H, bool FOLD_X>
__device__ __forceinline__ void finish_pair(const FinishParams& p, uint32_t tmem_row, int buf, float4 st,
                                            uint8_t* stg, int r) {
  const float2 rz = make_float2(st.x, st.x), nz = make_float2(st.y, st.y);
  const float2 rx = FOLD_X ? make_float2(st.z, st.z) : make_float2(p.inv_scale_o, p.inv_scale_o);
  const float2 nx = make_float2(st.w, st.w);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int o0 = 64 * H + cc * 16;
    uint32_t yv[16], gv[16];
    tmem_ld16(tmem_row + (uint32_t)(buf * 2 * kC + o0), yv);
    tmem_ld16(tmem_row + (uint32_t)(buf * 2 * kC + kC + o0), gv);
    tmem_ld_wait();
    uint32_t packed[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int o = o0 + e;
      // W_o', its constants, W_g' and the gate constants all carry a factor 1/2 (exact), so that
      // hy = y / 2 and hg = g / 2, and y * sigmoid(g) = hy + hy * tanh(hg): one MUFU operation.
      const float2 bo = make_float2(p.cst[2 * kC + o], p.cst[2 * kC + o + 1]);
      const float2 hy = __ffma2_rn(rx, make_float2(__uint_as_float(yv[e]), __uint_as_float(yv[e + 1])),
                                   FOLD_X ? __ffma2_rn(nx, make_float2(p.cst[3 * kC + o], p.cst[3 * kC + o + 1]), bo)
                                          : bo);
      const float2 hg = __ffma2_rn(rz, make_float2(__uint_as_float(gv[e]), __uint_as_float(gv[e + 1])),
                                   __ffma2_rn(nz, make_float2(p.cst[o], p.cst[o + 1]),
                                              make_float2(p.cst[kC + o], p.cst[kC + o + 1])));
      const float2 v = __ffma2_rn(hy, make_float2(tanh_mufu(hg.x), tanh_mufu(hg.y)), hy);
      packed[e >> 1] = pack_bf16x2(v.x, v.y);
    }
    // 16-byte units 2cc and 2cc + 1 of this pair's 128-byte staging row
    *reinterpret_cast<uint4*>(stg + sw128_offset(r, 2 * cc)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    *reinterpret_cast<uint4*>(stg + sw128_offset(r, 2 * cc + 1)) =
        make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}

__device__ __forceinline__ void load_weights(const Smem& sm, const CUtensorMap* womap, const CUtensorMap* wgmap) {
  mbar_expect_tx(&sm.bars->wfull, WO_BYTES + WG_BYTES);
  for (int kc = 0; kc < 2; ++kc) tma_load_2d(sm.wo + kc * (WO_BYTES / 2), womap, &sm.bars->wfull, kc * 64, 0);
  for (int hl = 0; hl < 2; ++hl)
    for (int kc = 0; kc < 2; ++kc)
      tma_load_2d(sm.wg + (hl * 2 + kc) * (WO_BYTES / 2), wgmap, &sm.bars->wfull, kc * 64, hl * kC);
}

// The epilogue role, shared by both kernels. The statistics buffer is handed back as soon as it has
// been read. X16: the staging box is the epilogue's own; float32: it is the x-hat buffer, handed
// back to the LayerNorm warps through hempty once the stores have read it.
template <bool X16>
__device__ __forceinline__ void epilogue_role(const FinishParams& p, const Smem& sm, uint32_t tmem_base,
                                              const CUtensorMap* omap, volatile int* abort_flag, int warp,
                                              int lane) {
  Bars& b = *sm.bars;
  const int ew = warp - 2 - LN_WARPS;      // 0..7
  const int q = warp & 3;                  // TMEM lane quadrant: pairs 32q .. 32q+31
  const int r = q * 32 + lane;
  const int hsel = ew >> 2;                // output channels 64*hsel .. 64*hsel + 63
  const uint32_t tmem_row = tmem_base + ((uint32_t)(q * 32) << 16);
  uint8_t* stg = sm.xh + hsel * (XH_BYTES / 2);
  int local = 0;
  for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
    const int il = (int)(t / p.tiles_j);
    const int jt = (int)(t - (long long)il * p.tiles_j);
    const int buf = local & 1;
    const uint32_t use = (uint32_t)(local >> 1);
    // X16: LayerNorm_in statistics of this thread's pair, as the projection kernel left them; the load
    // is issued before the waits so that its latency hides behind them
    float2 zst = make_float2(0.f, 0.f);
    if (X16 && jt * BM + r < p.bj) zst = p.zstat[(size_t)(p.i0 + il) * p.N + (p.j0 + jt * BM + r)];
    if (!warp_wait_bounded(&b.sfull[0], (uint32_t)local & 1u, p.w, abort_flag, 43)) break;
    if (!warp_wait_bounded(&b.tfull[buf], use & 1u, p.w, abort_flag, 41)) break;
    tc_fence_after();
    float4 st = sm.st[r];
    if (X16) {
      st.x = zst.x;
      st.y = zst.y;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&b.sempty[0]);     // the statistics of this tile have been read
    if (X16) {
      if (lane == 0) bulk_wait_read<0>();          // this warp's previous store has read its rows
      __syncwarp();
    }
    if (hsel == 0)
      finish_pair<0, X16>(p, tmem_row, buf, st, stg, r);
    else
      finish_pair<1, X16>(p, tmem_row, buf, st, stg, r);
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&b.tempty[buf]);
      // rows 32q .. 32q+31 of the box: one TMA store (pairs past the block's edge are clipped by the
      // map, whose extents are the block's)
      // (residual: the box is added to out, which holds z: out = z + update, rounded once to bf16 where
      // it lands)
      if (jt * BM + q * 32 < p.bj) {
        if (p.residual)
          tma_reduce_add_3d(omap, stg + q * 32 * 128, hsel * 64, jt * BM + q * 32, il);
        else
          tma_store_3d(omap, stg + q * 32 * 128, hsel * 64, jt * BM + q * 32, il);
        bulk_commit();
      }
      if (!X16) {
        bulk_wait_read<0>();
        mbar_arrive(&b.hempty);
      }
    }
  }
  if (lane == 0) bulk_wait_all();   // stores out before the CTA's shared memory goes away
}

__device__ __forceinline__ void init_common(const Smem& sm, uint32_t xempty_count, uint32_t zempty_count,
                                            uint32_t s_count, const FinishParams& p) {
  Bars& b = *sm.bars;
  b.abort_flag = (smem_u32(sm.zs) & 1023u) ? 1 : 0;
  if (b.abort_flag) raise_status(p.w, ST_TIMEOUT, 90);
  for (int i = 0; i < 2; ++i) {
    mbar_init(&b.xfull[i], 1);
    mbar_init(&b.xempty[i], xempty_count);
    mbar_init(&b.tfull[i], 1);
    mbar_init(&b.tempty[i], EPI_WARPS);
    mbar_init(&b.sfull[i], LN_WARPS);
    mbar_init(&b.sempty[i], s_count);
  }
  mbar_init(&b.zfull, 1);
  mbar_init(&b.zempty, zempty_count);
  mbar_init(&b.hfull, LN_WARPS);
  mbar_init(&b.hempty, EPI_WARPS);
  mbar_init(&b.wfull, 1);
  mbar_init(&b.fin, 1);
  fence_mbar_init();
}

__device__ __forceinline__ void teardown(const Smem& sm, uint32_t tmem_base, int warp) {
  __syncthreads();
  if (sm.bars->abort_flag) {
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 2000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ================================================================== fp16 x, folded LayerNorm
__global__ void __launch_bounds__(THREADS, 1)
    k3_finish_x16(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap zmap,
                  const __grid_constant__ CUtensorMap womap, const __grid_constant__ CUtensorMap wgmap,
                  const __grid_constant__ CUtensorMap omap, const __grid_constant__ FinishParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem sm(smem);
  Bars& b = *sm.bars;
  volatile int* abort_flag = &b.abort_flag;
  constexpr int SLOT = XS_BYTES / 2;        // one fp16 x tile: two 64-pair boxes of [128 c][64 j]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // x slots are released by the MMA and the statistics warps, z by the MMA alone (z's LayerNorm
  // statistics come from the projection kernel); the statistics buffer by the epilogue warps
  if (threadIdx.x == 0) init_common(sm, 1 + LN_WARPS, 1, EPI_WARPS, p);
  if (warp == 1) {
    tmem_alloc(&b.tslot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = b.tslot;

  if (!*abort_flag) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&zmap);
        load_weights(sm, &womap, &wgmap);
        uint32_t ph = 0;
        int local = 0;
        for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
          const int il = (int)(t / p.tiles_j);
          const int jt = (int)(t - (long long)il * p.tiles_j);
          const int xsl = local & 1;
          if (!wait_bounded(&b.xempty[xsl], ((uint32_t)(local >> 1) & 1u) ^ 1u, p.w, abort_flag, 31)) break;
          mbar_expect_tx(&b.xfull[xsl], SLOT);
          uint8_t* slot = sm.xs + xsl * SLOT;
          tma_load_3d(slot, &xmap, &b.xfull[xsl], jt * BM, il, 0);
          tma_load_3d(slot + SLOT / 2, &xmap, &b.xfull[xsl], jt * BM + 64, il, 0);
          if (!wait_bounded(&b.zempty, ph ^ 1u, p.w, abort_flag, 32)) break;
          mbar_expect_tx(&b.zfull, Z_BYTES);
          tma_load_3d(sm.zs, &zmap, &b.zfull, 0, p.j0 + jt * BM, p.i0 + il);
          tma_load_3d(sm.zs + Z_BYTES / 2, &zmap, &b.zfull, 64, p.j0 + jt * BM, p.i0 + il);
          {
            // the next tile's z into L2 now: its load waits for this tile's MMAs (one z stage), and
            // then finds it there instead of in HBM
            const long long tn = t + gridDim.x;
            if (tn < p.total_tiles) {
              const int iln = (int)(tn / p.tiles_j);
              const int jtn = (int)(tn - (long long)iln * p.tiles_j);
              tma_prefetch_l2_3d(&zmap, 0, p.j0 + jtn * BM, p.i0 + iln);
              tma_prefetch_l2_3d(&zmap, 64, p.j0 + jtn * BM, p.i0 + iln);
            }
          }
          ph ^= 1u;
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        // y: A = x16 tile, M-major (pairs contiguous); B = W_o' K-major. g: A = z, B = W_g' hi, lo.
        constexpr uint32_t id_y = make_idesc(BM, kC, FMT_F16, true, false);
        constexpr uint32_t id_g = make_idesc(BM, kC, FMT_BF16, false, false);
        uint32_t ph = 0;
        int local = 0;
        if (wait_bounded(&b.wfull, 0, p.w, abort_flag, 33)) {
          // operand descriptors formed once; per MMA the tile's descriptor plus the byte offset / 16
          // (the start-address field, shared memory below 256 KB)
          const uint64_t dz = make_sdesc_sw128(smem_u32(sm.zs), 16, 1024);
          const uint64_t dwo = make_sdesc_sw128(smem_u32(sm.wo), 16, 1024);
          const uint64_t dwg = make_sdesc_sw128(smem_u32(sm.wg), 16, 1024);
          const uint64_t dx = make_sdesc_sw128(smem_u32(sm.xs), SLOT / 2, 1024);
          for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            const int xsl = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!wait_bounded(&b.tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 34)) break;
            if (!wait_bounded(&b.xfull[xsl], use & 1u, p.w, abort_flag, 35)) break;
            if (!wait_bounded(&b.zfull, ph, p.w, abort_flag, 36)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(buf * 2 * kC);
            const uint64_t dxs = dx + (uint32_t)((xsl * SLOT) >> 4);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              // x: 16 channel rows of 128 bytes per K step; the two 64-pair halves are SLOT/2 apart
              const uint32_t woff = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
              mma_f16(d, dxs + (uint32_t)((ks * 2048) >> 4), dwo + woff, id_y, ks != 0);
              mma_f16(d + kC, dz + woff, dwg + woff, id_g, ks != 0);
              mma_f16(d + kC, dz + woff, dwg + ((2u * 16384u) >> 4) + woff, id_g, 1u);
            }
            mma_commit(&b.xempty[xsl]);
            mma_commit(&b.zempty);
            mma_commit(&b.tfull[buf]);
            ph ^= 1u;
          }
        }
        mma_commit(&b.fin);
        wait_bounded(&b.fin, 0, p.w, abort_flag, 37);
      }
    } else if (warp < 2 + LN_WARPS) {
      // ------------------------------------------------------------ statistics, two lanes per pair
      // Lane l of warp w takes channel half hc = l / 16: x columns p0 = 32w + 2 (l % 16) and p0 + 1
      // (one 4-byte load covers both; fp32x2 math over the two pairs).
      const int lw = warp - 2;
      const int lp = lane & 15, hc = lane >> 4;
      const int p0 = lw * 32 + 2 * lp;
      // x16[c][p0], [c][p0 + 1] in a slot: the 64-pair half, 16-byte unit and byte of the pair
      const int xoff = (p0 >> 6) * (SLOT / 2) + ((p0 & 7) << 1);
      const uint32_t xunit = (uint32_t)((p0 & 63) >> 3);
      // LayerNorm epsilon in the units x16 = x 2^e is stored in
      const float x_eps = 1e-5f * __int_as_float((127 + 2 * p.x_exp) << 23);
      int local = 0;
      for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
        const int xsl = local & 1;
        if (!warp_wait_bounded(&b.xfull[xsl], (uint32_t)(local >> 1) & 1u, p.w, abort_flag, 39)) break;
        const uint8_t* xrow = sm.xs + xsl * SLOT + xoff;
        auto ld = [&](int c) {
          return __half22float2(*reinterpret_cast<const __half2*>(xrow + sw128_offset((uint32_t)c, xunit)));
        };
        const int cb = hc * 64;
        const float2 sh = ld(cb);
        const float2 nsh = make_float2(-sh.x, -sh.y);
        float2 s0 = make_float2(0.f, 0.f), s1 = s0, q0 = s0, q1 = s0;
#pragma unroll 8
        for (int c = 0; c < 64; c += 2) {
          const float2 d0 = __fadd2_rn(ld(cb + c), nsh), d1 = __fadd2_rn(ld(cb + c + 1), nsh);
          s0 = __fadd2_rn(s0, d0);
          s1 = __fadd2_rn(s1, d1);
          q0 = __ffma2_rn(d0, d0, q0);
          q1 = __ffma2_rn(d1, d1, q1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.xempty[xsl]);   // this warp is done reading the x slot
        const float2 ss = __fadd2_rn(s0, s1), vs = __fadd2_rn(q0, q1);
        float xm0, xr0, xm1, xr1;
        merge_halves(sh.x + ss.x * (1.0f / 64), vs.x - ss.x * ss.x * (1.0f / 64), x_eps, xm0, xr0);
        merge_halves(sh.y + ss.y * (1.0f / 64), vs.y - ss.y * ss.y * (1.0f / 64), x_eps, xm1, xr1);
        // the epilogue has read the previous tile's statistics
        if (!warp_wait_bounded(&b.sempty[0], ((uint32_t)local & 1u) ^ 1u, p.w, abort_flag, 42)) break;
        float2* st2 = reinterpret_cast<float2*>(sm.st);
        // lane hc of the two that share the pairs writes pair p0 + hc. rx carries the scale of W_o'
        // (1/2 and its power of two): y/2 = rx acc + nx rowsum' + bias'.
        st2[2 * (p0 + hc) + 1] = hc ? make_float2(p.inv_scale_o * xr1, -xr1 * xm1)
                                    : make_float2(p.inv_scale_o * xr0, -xr0 * xm0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.sfull[0]);
      }
    } else {
      epilogue_role<true>(p, sm, tmem_base, &omap, abort_flag, warp, lane);
    }
  }
  teardown(sm, tmem_base, warp);
}

// ================================================================== float32 x, x-hat operand
__global__ void __launch_bounds__(THREADS, 1)
    k3_finish_x32(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap zmap,
                  const __grid_constant__ CUtensorMap womap, const __grid_constant__ CUtensorMap wgmap,
                  const __grid_constant__ CUtensorMap omap, const __grid_constant__ FinishParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem sm(smem);
  Bars& b = *sm.bars;
  volatile int* abort_flag = &b.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) init_common(sm, LN_WARPS, 1, EPI_WARPS, p);
  if (warp == 1) {
    tmem_alloc(&b.tslot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = b.tslot;

  if (!*abort_flag) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&zmap);
        load_weights(sm, &womap, &wgmap);
        uint32_t ph = 0;
        for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
          const int il = (int)(t / p.tiles_j);
          const int jt = (int)(t - (long long)il * p.tiles_j);
          if (!wait_bounded(&b.xempty[0], ph ^ 1u, p.w, abort_flag, 31)) break;
          mbar_expect_tx(&b.xfull[0], XS_BYTES);
          tma_load_3d(sm.xs, &xmap, &b.xfull[0], jt * BM, il, 0);
          if (!wait_bounded(&b.zempty, ph ^ 1u, p.w, abort_flag, 32)) break;
          mbar_expect_tx(&b.zfull, Z_BYTES);
          tma_load_3d(sm.zs, &zmap, &b.zfull, 0, p.j0 + jt * BM, p.i0 + il);
          tma_load_3d(sm.zs + Z_BYTES / 2, &zmap, &b.zfull, 64, p.j0 + jt * BM, p.i0 + il);
          {
            // the next tile's z into L2 now: its load waits for this tile's MMAs (one z stage), and
            // then finds it there instead of in HBM
            const long long tn = t + gridDim.x;
            if (tn < p.total_tiles) {
              const int iln = (int)(tn / p.tiles_j);
              const int jtn = (int)(tn - (long long)iln * p.tiles_j);
              tma_prefetch_l2_3d(&zmap, 0, p.j0 + jtn * BM, p.i0 + iln);
              tma_prefetch_l2_3d(&zmap, 64, p.j0 + jtn * BM, p.i0 + iln);
            }
          }
          ph ^= 1u;
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_y = make_idesc(BM, kC, FMT_F16, false, false);
        constexpr uint32_t id_g = make_idesc(BM, kC, FMT_BF16, false, false);
        uint32_t ph = 0;
        int local = 0;
        if (wait_bounded(&b.wfull, 0, p.w, abort_flag, 33)) {
          // operand descriptors formed once; per MMA the tile's descriptor plus the byte offset / 16
          const uint64_t dh = make_sdesc_sw128(smem_u32(sm.xh), 16, 1024);
          const uint64_t dz = make_sdesc_sw128(smem_u32(sm.zs), 16, 1024);
          const uint64_t dwo = make_sdesc_sw128(smem_u32(sm.wo), 16, 1024);
          const uint64_t dwg = make_sdesc_sw128(smem_u32(sm.wg), 16, 1024);
          for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!wait_bounded(&b.tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 34)) break;
            if (!wait_bounded(&b.hfull, ph, p.w, abort_flag, 35)) break;
            if (!wait_bounded(&b.zfull, ph, p.w, abort_flag, 36)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(buf * 2 * kC);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
              mma_f16(d, dh + off, dwo + off, id_y, ks != 0);
              mma_f16(d + kC, dz + off, dwg + off, id_g, ks != 0);
              mma_f16(d + kC, dz + off, dwg + ((2u * 16384u) >> 4) + off, id_g, 1u);
            }
            mma_commit(&b.zempty);
            mma_commit(&b.tfull[buf]);
            ph ^= 1u;
          }
        }
        mma_commit(&b.fin);
        wait_bounded(&b.fin, 0, p.w, abort_flag, 37);
      }
    } else if (warp < 2 + LN_WARPS) {
      // ------------------------------------------------------------ LayerNorm, two lanes per pair
      // As in the fp16 kernel (x columns p0, p0 + 1, channel half hc; z rows zr0, zr0 + 16), with a
      // second pass over the float32 x that writes the normalised fp16 rows of a K-major operand.
      const int lw = warp - 2;
      const int lp = lane & 15, hc = lane >> 4;
      const int p0 = lw * 32 + 2 * lp;
      const int zr0 = lw * 32 + lp;
      const int cb = hc * 64;
      uint32_t ph = 0;
      int local = 0;
      for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
        if (!warp_wait_bounded(&b.zfull, ph, p.w, abort_flag, 38)) break;
        float zmean[2], zrstd[2];
        z_stats(sm.zs, zr0, hc, zmean, zrstd);
        // the epilogue has read the previous tile's statistics
        if (!warp_wait_bounded(&b.sempty[0], ((uint32_t)local & 1u) ^ 1u, p.w, abort_flag, 42)) break;
        reinterpret_cast<float2*>(sm.st)[2 * (zr0 + 16 * hc)] =
            hc ? make_float2(zrstd[1], -zrstd[1] * zmean[1]) : make_float2(zrstd[0], -zrstd[0] * zmean[0]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&b.sfull[0]);

        if (!warp_wait_bounded(&b.xfull[0], ph, p.w, abort_flag, 39)) break;
        const float* xcol = reinterpret_cast<const float*>(sm.xs) + cb * BM + p0;
        auto xpair = [&](int c) { return *reinterpret_cast<const float2*>(xcol + c * BM); };
        const float2 xsh = xpair(0);
        const float2 nxsh = make_float2(-xsh.x, -xsh.y);
        float2 s0 = make_float2(0.f, 0.f), s1 = s0, v0 = s0, v1 = s0;
#pragma unroll 8
        for (int c = 0; c < 64; c += 2) {
          const float2 d0 = __fadd2_rn(xpair(c), nxsh);
          const float2 d1 = __fadd2_rn(xpair(c + 1), nxsh);
          s0 = __fadd2_rn(s0, d0);
          s1 = __fadd2_rn(s1, d1);
          v0 = __ffma2_rn(d0, d0, v0);
          v1 = __ffma2_rn(d1, d1, v1);
        }
        const float2 ss = __fadd2_rn(s0, s1), vs = __fadd2_rn(v0, v1);
        float xm0, xr0, xm1, xr1;
        merge_halves(xsh.x + ss.x * (1.0f / 64), vs.x - ss.x * ss.x * (1.0f / 64), 1e-5f, xm0, xr0);
        merge_halves(xsh.y + ss.y * (1.0f / 64), vs.y - ss.y * ss.y * (1.0f / 64), 1e-5f, xm1, xr1);
        const float2 xr2 = make_float2(xr0, xr1), xb2 = make_float2(-xr0 * xm0, -xr1 * xm1);
        if (!warp_wait_bounded(&b.hempty, ph ^ 1u, p.w, abort_flag, 40)) break;
        uint8_t* xhc = sm.xh + hc * (XH_BYTES / 2);
#pragma unroll 2
        for (int u = 0; u < 8; ++u) {
          // 16-byte unit uu (channels 64 hc + 8 uu ..) of rows p0 and p0 + 1; the unit order is
          // rotated by lane group so that the 16 lanes of a half store to distinct bank groups
          const int uu = (u + (lp >> 2)) & 7;
          uint32_t h0[4], h1[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 e0 = __ffma2_rn(xpair(8 * uu + 2 * k), xr2, xb2);
            const float2 e1 = __ffma2_rn(xpair(8 * uu + 2 * k + 1), xr2, xb2);
            h0[k] = pack_f16x2(e0.x, e1.x);
            h1[k] = pack_f16x2(e0.y, e1.y);
          }
          *reinterpret_cast<uint4*>(xhc + sw128_offset(p0, uu)) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
          *reinterpret_cast<uint4*>(xhc + sw128_offset(p0 + 1, uu)) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&b.xempty[0]);
          mbar_arrive(&b.hfull);
        }
        ph ^= 1u;
      }
    } else {
      epilogue_role<false>(p, sm, tmem_base, &omap, abort_flag, warp, lane);
    }
  }
  teardown(sm, tmem_base, warp);
}

}  // namespace

cudaError_t launch_finish_bf16(bool x16, const CUtensorMap& xmap, const CUtensorMap& zmap,
                               const CUtensorMap& womap, const CUtensorMap& wgmap, const CUtensorMap& omap,
                               const FinishParams& p, int num_sms, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  cudaError_t err = once_per_device(attr_set, [] {
    cudaError_t e = cudaFuncSetAttribute(k3_finish_x16, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k3_finish_x32, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (err != cudaSuccess) return err;
  if (p.total_tiles <= 0) return cudaSuccess;
  const int grid = (int)(p.total_tiles < num_sms ? p.total_tiles : num_sms);
  if (x16)
    k3_finish_x16<<<grid, THREADS, SMEM_BYTES, s>>>(xmap, zmap, womap, wgmap, omap, p);
  else
    k3_finish_x32<<<grid, THREADS, SMEM_BYTES, s>>>(xmap, zmap, womap, wgmap, omap, p);
  return cudaGetLastError();
}

}  // namespace tmk
