// k3_finish.cu -- output stage of the triangle multiplicative update on the
// sm_103a tensor cores, over one output block:
//
//   out_ij = sigmoid(W_g zh_ij) * W_o LayerNorm_out(x_ij),   zh = LayerNorm_in(z)
//
// x comes channel-major [128][bi][ldx] from the contraction, float32 or fp16
// scaled by 2^e (LayerNorm is scale-free apart from its epsilon, which is
// scaled to match, so the fp16 values are normalised as they are); z and out
// are the caller's bf16 [N][N][128] pair representation (the layer(x, mask)
// call of the code-sample section of "NVIDIA BioNeMo escala modelagem
// biomolecular com context parallelism e quebra barreira de memória da GPU").
//
// Per tile of 128 pairs (one row i, 128 consecutive j of the block):
//   warp 0      TMA: x tile [128 c][128 j], fp16 (32 KB, two tiles in flight) or
//               float32 (64 KB, one), z tile (two 64-channel boxes, 128-byte
//               swizzle); W_o (fp16) and W_g (bf16 hi + lo) once.
//   warps 2..5  LayerNorm, two lanes per pair (one per channel half): a shifted
//               one-pass sum and sum of squares per half, merged across the two
//               lanes, then a normalising pass that writes the fp16 rows of a
//               K-major operand; 8-byte loads cover two pairs at a time. z's
//               statistics the same way, handed to the epilogue through a
//               double-buffered shared array behind mbarriers. The producer
//               also prefetches the next two tiles' boxes into L2.
//   warp 1      tcgen05.mma: D[p][0..128) = xh x W_o'^T (kind::f16, fp16),
//               D[p][128..256) = z x W_g'^T (bf16, hi and lo), two TMEM buffers.
//   warps 6..13 epilogue, thread = pair: two warps per TMEM lane quadrant split
//               the 128 output channels; gate (sigmoid through one tanh) and
//               product, staged in the x-hat buffer (free once the tile's MMA has
//               read it) and written by one TMA store of 32 pairs x 64 channels
//               per warp; the buffer goes back to the LayerNorm warps when the
//               stores have read it.
// LayerNorm_out's gamma is folded into W_o' = W_o diag(gamma_out) (scaled by a
// power of two to use fp16's range) and beta into a bias; LayerNorm_in of the
// gate is folded as in the projection: W_g zh = rstd (W_g' z - mu rowsum) + bias.
// The per-channel constants travel in the kernel's parameter block.
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int BM = kFinishTileJ;             // pairs per tile
constexpr int XS_BYTES = kC * BM * 4;        // x staging: one fp32 [c][j] tile or two fp16 ones (64 KB)
constexpr int XH_BYTES = BM * kC * 2;        // 32 KB fp16, two K-chunks
constexpr int Z_BYTES = BM * kC * 2;         // 32 KB bf16, two K-chunks
constexpr int WO_BYTES = kC * kC * 2;        // 32 KB fp16
constexpr int WG_BYTES = 2 * kC * kC * 2;    // 64 KB bf16 hi + lo
constexpr int LN_WARPS = 4, EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * (LN_WARPS + EPI_WARPS);
constexpr int ZST_BYTES = 2 * BM * 8;        // two buffers of float2 (rstd, -rstd*mu) per pair
// mbarriers and flags, after the tiles
struct Bars {
  uint64_t xfull[2], xempty[2];   // x ring (fp16: two slots; float32: slot 0 only)
  uint64_t zfull, zempty;         // z tile
  uint64_t hfull, hempty;         // x-hat operand / out staging
  uint64_t tfull[2], tempty[2];   // TMEM accumulators
  uint64_t sfull[2], sempty[2];   // z statistics
  uint64_t wfull, fin;
  uint32_t tslot;
  int abort_flag;
};
constexpr int SMEM_BYTES = XS_BYTES + XH_BYTES + Z_BYTES + WO_BYTES + WG_BYTES + ZST_BYTES + 256;
static_assert(sizeof(Bars) <= 256, "barrier block");
constexpr int TMEM_COLS = 512;

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(kBoxFinishX.bytes() == XS_BYTES && 2 * kBoxFinishX16.bytes() == XS_BYTES, "x tiles = one box each");
static_assert(2 * kBoxFinishZ.bytes() == Z_BYTES, "z tile = two boxes");
static_assert(2 * kBoxFinishW.bytes() == WO_BYTES && 4 * kBoxFinishW.bytes() == WG_BYTES, "weight boxes");
static_assert(EPI_WARPS * kBoxFinishOut.bytes() == XH_BYTES && kBoxFinishOut.d0 * 2 == 128,
              "out staging: one 32-row box of 128-byte rows per epilogue warp fills the x-hat buffer");

__device__ __forceinline__ float2 bf2f(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// Epilogue of one tile for one thread: pair row of the TMEM accumulator at `tmem_row`, output
// channels [64*H, 64*H + 64), written as bf16 into row `r` of the 128-byte-swizzled staging box
// `stg` (64 channels x 128 pairs, the K-major layout of the x-hat operand whose buffer it reuses).
// H is a template parameter so the constant-bank offsets are immediates.
template <int H>
__device__ __forceinline__ void finish_pair(const FinishParams& p, uint32_t tmem_row, int buf, float2 zst,
                                            uint8_t* stg, int r) {
  const float2 inv = make_float2(p.inv_scale_o, p.inv_scale_o);
  const float2 r2 = make_float2(zst.x, zst.x), n2 = make_float2(zst.y, zst.y);
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
      // W_o', its bias, W_g' and the gate constants all carry a factor 1/2 (exact), so that
      // hy = y / 2 and hg = g / 2, and y * sigmoid(g) = hy + hy * tanh(hg): one MUFU operation.
      const float2 hy = __ffma2_rn(make_float2(__uint_as_float(yv[e]), __uint_as_float(yv[e + 1])), inv,
                                   make_float2(p.cst[2 * kC + o], p.cst[2 * kC + o + 1]));
      const float2 hg = __ffma2_rn(r2, make_float2(__uint_as_float(gv[e]), __uint_as_float(gv[e + 1])),
                                   __ffma2_rn(n2, make_float2(p.cst[o], p.cst[o + 1]),
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

// X16: x arrives as fp16 (scaled by 2^e, e from the projection's maxima), two tiles in flight;
// otherwise as float32, one tile at a time.
template <bool X16>
__global__ void __launch_bounds__(THREADS, 1)
    k3_finish(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap zmap,
              const __grid_constant__ CUtensorMap womap, const __grid_constant__ CUtensorMap wgmap,
              const __grid_constant__ CUtensorMap omap, const __grid_constant__ FinishParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* zs = smem;                        // 1024-aligned swizzled tiles first
  uint8_t* xh = zs + Z_BYTES;
  uint8_t* wo = xh + XH_BYTES;
  uint8_t* wg = wo + WO_BYTES;               // hi chunks then lo chunks
  uint8_t* xs = wg + WG_BYTES;              // float32 [c][j], or two fp16 [c][j] slots
  float2* zst = reinterpret_cast<float2*>(xs + XS_BYTES);   // [2][128]: rstd_z, -rstd_z * mu_z
  Bars& bars = *reinterpret_cast<Bars*>(zst + 2 * BM);
  uint64_t* xfull = bars.xfull;
  uint64_t* xempty = bars.xempty;
  uint64_t* zfull = &bars.zfull;
  uint64_t* zempty = &bars.zempty;
  uint64_t* hfull = &bars.hfull;
  uint64_t* hempty = &bars.hempty;
  uint64_t* tfull = bars.tfull;
  uint64_t* tempty = bars.tempty;
  uint64_t* sfull = bars.sfull;
  uint64_t* sempty = bars.sempty;
  uint64_t* wfull = &bars.wfull;
  uint64_t* fin = &bars.fin;
  uint32_t* tslot = &bars.tslot;
  volatile int* abort_flag = &bars.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
    if (*abort_flag) raise_status(p.w, ST_TIMEOUT, 90);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], 1);
      // fp16: the slot holds x-hat after x, and is free once the MMA has read it; float32: once
      // the LayerNorm warps have read x (x-hat has its own buffer)
      mbar_init(&xempty[b], X16 ? 1 : LN_WARPS);
    }
    mbar_init(zfull, 1);
    mbar_init(zempty, X16 ? 1 + LN_WARPS : 1);   // fp16: the LayerNorm warps read z after x-hat
    mbar_init(hfull, LN_WARPS);
    mbar_init(hempty, EPI_WARPS);         // the epilogue's stores have read their staging rows
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EPI_WARPS);
      mbar_init(&sfull[b], LN_WARPS);
      mbar_init(&sempty[b], EPI_WARPS);
    }
    mbar_init(wfull, 1);
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tslot;

  if (!*abort_flag) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&zmap);
        mbar_expect_tx(wfull, WO_BYTES + WG_BYTES);
        for (int kc = 0; kc < 2; ++kc) tma_load_2d(wo + kc * (WO_BYTES / 2), &womap, wfull, kc * 64, 0);
        for (int hl = 0; hl < 2; ++hl)
          for (int kc = 0; kc < 2; ++kc)
            tma_load_2d(wg + (hl * 2 + kc) * (WO_BYTES / 2), &wgmap, wfull, kc * 64, hl * kC);
        constexpr uint32_t XT_BYTES = X16 ? kBoxFinishX16.bytes() : kBoxFinishX.bytes();
        uint32_t ph = 0;
        int local = 0;
        for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
          const int il = (int)(t / p.tiles_j);
          const int jt = (int)(t - (long long)il * p.tiles_j);
          // x ring: two fp16 slots used alternately, or the one float32 slot
          const int xsl = X16 ? (local & 1) : 0;
          const uint32_t xph = X16 ? (uint32_t)(local >> 1) & 1u : ph;
          if (!wait_bounded(&xempty[xsl], xph ^ 1u, p.w, abort_flag, 31)) break;
          mbar_expect_tx(&xfull[xsl], XT_BYTES);
          tma_load_3d(xs + xsl * (XS_BYTES / 2), &xmap, &xfull[xsl], jt * BM, il, 0);
          if (!wait_bounded(zempty, ph ^ 1u, p.w, abort_flag, 32)) break;
          mbar_expect_tx(zfull, Z_BYTES);
          tma_load_3d(zs, &zmap, zfull, 0, p.j0 + jt * BM, p.i0 + il);
          tma_load_3d(zs + Z_BYTES / 2, &zmap, zfull, 64, p.j0 + jt * BM, p.i0 + il);
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
        if (wait_bounded(wfull, 0, p.w, abort_flag, 33)) {
          const uint32_t z0 = smem_u32(zs), o0 = smem_u32(wo), g0 = smem_u32(wg);
          for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!wait_bounded(&tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 34)) break;
            if (!wait_bounded(hfull, ph, p.w, abort_flag, 35)) break;
            if (!wait_bounded(zfull, ph, p.w, abort_flag, 36)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(buf * 2 * kC);
            // x-hat: in this tile's x slot (fp16 x) or in its own buffer (float32 x)
            const uint32_t h0 = X16 ? smem_u32(xs + (local & 1) * (XS_BYTES / 2)) : smem_u32(xh);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint32_t off = kc * 16384 + ks * 32;
                mma_f16(d, make_sdesc_sw128(h0 + off, 16, 1024), make_sdesc_sw128(o0 + off, 16, 1024), id_y,
                        (kc | ks) != 0);
                mma_f16(d + kC, make_sdesc_sw128(z0 + off, 16, 1024), make_sdesc_sw128(g0 + off, 16, 1024), id_g,
                        (kc | ks) != 0);
                mma_f16(d + kC, make_sdesc_sw128(z0 + off, 16, 1024),
                        make_sdesc_sw128(g0 + 2 * 16384 + off, 16, 1024), id_g, 1u);
              }
            if (X16) mma_commit(&xempty[local & 1]);
            mma_commit(zempty);
            mma_commit(&tfull[buf]);
            ph ^= 1u;
          }
        }
        mma_commit(fin);
        wait_bounded(fin, 0, p.w, abort_flag, 37);
      }
    } else if (warp < 2 + LN_WARPS) {
      // ------------------------------------------------------------ LayerNorm, two lanes per pair
      // Lane l of LayerNorm warp w takes channel half hc = l / 16 of pair group 32w .. 32w+31:
      // x columns p0 = 32w + 2 (l % 16) and p0 + 1 (one load along j covers both, fp32x2 math over
      // the two pairs), z rows 32w + l % 16 and that + 16. Each half gives a shifted one-pass mean and sum of
      // squared deviations of its 64 channels; the two halves meet through a lane exchange and are
      // merged with the pairwise update of the mean and the sum of squares (Chan, Golub, LeVeque).
      const int lw = warp - 2;
      const int lp = lane & 15, hc = lane >> 4;
      const int p0 = lw * 32 + 2 * lp;
      const int zr0 = lw * 32 + lp;
      const int cb = hc * 64;
      // mean and variance of 128 channels from the two halves' (mean, M2) over 64 channels each
      auto merge = [](float mean_h, float m2_h, float eps, float& mean, float& rstd) {
        const float mean_o = __shfl_xor_sync(0xffffffffu, mean_h, 16);
        const float m2_o = __shfl_xor_sync(0xffffffffu, m2_h, 16);
        const float dm = mean_h - mean_o;
        mean = 0.5f * (mean_h + mean_o);
        const float var = fmaxf((m2_h + m2_o + 32.0f * dm * dm) * (1.0f / kC), 0.f);
        rstd = rsqrtf(var + eps);
      };
      // statistics of z over its 128 channels: rows zr0 and zr0 + 16, K-chunk hc of the tile
      auto z_stats = [&](float (&zmean)[2], float (&zrstd)[2]) {
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
          merge(sh + sd * (1.0f / 64), (qs.x + qs.y) - sd * sd * (1.0f / 64), 1e-5f, zmean[rr], zrstd[rr]);
        }
      };
      uint32_t ph = 0;
      int local = 0;
      if constexpr (X16) {
        // fp16 x, scaled by 2^e: LayerNorm reads the scaled values with epsilon scaled alike. Each
        // thread takes the statistics of its 64 channels x 2 pairs in one pass over shared memory,
        // builds their x-hat in registers in a second (a 2 x 2 transpose per channel pair) and, once
        // every LayerNorm thread has read the slot, writes x-hat over x in the same slot as the
        // K-major operand of the MMA.
        const int e = x16_exponent(p.amax, p.N);
        const float x_eps = 1e-5f * __int_as_float((127 + 2 * e) << 23);
        bool bad = false;
        for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
          const int sb = local & 1;
          const uint32_t sph = (uint32_t)(local >> 1) & 1u;
          const int xsl = local & 1;
          uint8_t* slot = xs + xsl * (XS_BYTES / 2);
          uint32_t v[64];
          if (!bad) bad = !warp_wait_bounded(&xfull[xsl], (uint32_t)(local >> 1) & 1u, p.w, abort_flag, 39);
          if (!bad) {
            // pass 1: statistics, straight from shared memory
            const __half* x16 = reinterpret_cast<const __half*>(slot) + cb * BM + p0;
            auto ld = [&](int c) { return __half22float2(*reinterpret_cast<const __half2*>(x16 + c * BM)); };
            const float2 sh = ld(0);
            const float2 nsh = make_float2(-sh.x, -sh.y);
            float2 s0 = make_float2(0.f, 0.f), s1 = s0, q0 = s0, q1 = s0;
#pragma unroll 8
            for (int c = 0; c < 64; c += 2) {
              const float2 d0 = __fadd2_rn(ld(c), nsh), d1 = __fadd2_rn(ld(c + 1), nsh);
              s0 = __fadd2_rn(s0, d0);
              s1 = __fadd2_rn(s1, d1);
              q0 = __ffma2_rn(d0, d0, q0);
              q1 = __ffma2_rn(d1, d1, q1);
            }
            const float2 ss = __fadd2_rn(s0, s1), vs = __fadd2_rn(q0, q1);
            float xm0, xr0, xm1, xr1;
            merge(sh.x + ss.x * (1.0f / 64), vs.x - ss.x * ss.x * (1.0f / 64), x_eps, xm0, xr0);
            merge(sh.y + ss.y * (1.0f / 64), vs.y - ss.y * ss.y * (1.0f / 64), x_eps, xm1, xr1);
            const float2 xr2 = make_float2(xr0, xr1), xb2 = make_float2(-xr0 * xm0, -xr1 * xm1);
            // pass 2: x-hat in registers, a 2 x 2 transpose per channel pair
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              const float2 e0 = __ffma2_rn(ld(c), xr2, xb2);       // channel c: pairs p0, p0 + 1
              const float2 e1 = __ffma2_rn(ld(c + 1), xr2, xb2);   // channel c + 1
              v[c] = pack_f16x2(e0.x, e1.x);                       // row p0: channels c, c + 1
              v[c + 1] = pack_f16x2(e0.y, e1.y);                   // row p0 + 1
            }
          }
          // every LayerNorm thread has read the slot before any thread overwrites it; a failed wait
          // anywhere stops all four warps here together
          if (named_bar_or(1, 32 * LN_WARPS, bad)) break;
          uint8_t* xhc = slot + hc * (XS_BYTES / 4);     // K-chunk hc of the x-hat operand
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            *reinterpret_cast<uint4*>(xhc + sw128_offset(p0, u)) =
                make_uint4(v[8 * u], v[8 * u + 2], v[8 * u + 4], v[8 * u + 6]);
            *reinterpret_cast<uint4*>(xhc + sw128_offset(p0 + 1, u)) =
                make_uint4(v[8 * u + 1], v[8 * u + 3], v[8 * u + 5], v[8 * u + 7]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(hfull);
          if (!bad) bad = !warp_wait_bounded(zfull, ph, p.w, abort_flag, 38);
          if (!bad) {
            float zmean[2], zrstd[2];
            z_stats(zmean, zrstd);
            __syncwarp();
            if (lane == 0) mbar_arrive(zempty);      // this warp is done reading the z tile
            bad = !warp_wait_bounded(&sempty[sb], sph ^ 1u, p.w, abort_flag, 42);
            if (!bad) {
              // lane hc of the two that share the rows writes row zr0 + 16 hc
              zst[sb * BM + zr0 + 16 * hc] = hc ? make_float2(zrstd[1], -zrstd[1] * zmean[1])
                                                : make_float2(zrstd[0], -zrstd[0] * zmean[0]);
              __syncwarp();
              if (lane == 0) mbar_arrive(&sfull[sb]);
            }
          }
          ph ^= 1u;
        }
      } else {
        const float x_eps = 1e-5f;
        for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
          const int sb = local & 1;
          const uint32_t sph = (uint32_t)(local >> 1) & 1u;
          if (!warp_wait_bounded(zfull, ph, p.w, abort_flag, 38)) break;
          float zmean[2], zrstd[2];
          z_stats(zmean, zrstd);
          if (!warp_wait_bounded(&sempty[sb], sph ^ 1u, p.w, abort_flag, 42)) break;
          // lane hc of the two that share the rows writes row zr0 + 16 hc
          zst[sb * BM + zr0 + 16 * hc] = hc ? make_float2(zrstd[1], -zrstd[1] * zmean[1])
                                            : make_float2(zrstd[0], -zrstd[0] * zmean[0]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfull[sb]);

          // float32 x: columns p0, p0 + 1 of the [c][j] tile, channels of half hc; two passes over
          // shared memory (statistics, then normalise into the x-hat buffer)
          if (!warp_wait_bounded(&xfull[0], ph, p.w, abort_flag, 39)) break;
          const float* xcol = reinterpret_cast<const float*>(xs) + cb * BM + p0;
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
          merge(xsh.x + ss.x * (1.0f / 64), vs.x - ss.x * ss.x * (1.0f / 64), x_eps, xm0, xr0);
          merge(xsh.y + ss.y * (1.0f / 64), vs.y - ss.y * ss.y * (1.0f / 64), x_eps, xm1, xr1);
          const float2 xr2 = make_float2(xr0, xr1), xb2 = make_float2(-xr0 * xm0, -xr1 * xm1);
          if (!warp_wait_bounded(hempty, ph ^ 1u, p.w, abort_flag, 40)) break;
          uint8_t* xhc = xh + hc * (XH_BYTES / 2);
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
            mbar_arrive(&xempty[0]);
            mbar_arrive(hfull);
          }
          ph ^= 1u;
        }
      }
    } else {
      // ------------------------------------------------------------ epilogue, thread = pair
      const int ew = warp - 2 - LN_WARPS;      // 0..7
      const int q = warp & 3;                  // TMEM lane quadrant: pairs 32q .. 32q+31
      const int r = q * 32 + lane;
      const int hsel = ew >> 2;                // output channels 64*hsel .. 64*hsel + 63
      const uint32_t tmem_row = tmem_base + ((uint32_t)(q * 32) << 16);
      int local = 0;
      for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
        const int il = (int)(t / p.tiles_j);
        const int jt = (int)(t - (long long)il * p.tiles_j);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        const int sb = local & 1;
        const uint32_t sph = (uint32_t)(local >> 1) & 1u;
        if (!warp_wait_bounded(&sfull[sb], sph, p.w, abort_flag, 43)) break;
        if (!warp_wait_bounded(&tfull[buf], use & 1u, p.w, abort_flag, 41)) break;
        tc_fence_after();
        const float2 zs2 = zst[sb * BM + r];
        // staging box of out: the x-hat buffer, free once this tile's MMA has read it (float32 x), or
        // that buffer kept for the epilogue alone (fp16 x, whose x-hat lives in the x slots)
        uint8_t* stg = xh + hsel * (XH_BYTES / 2);
        if (X16) {
          if (lane == 0) bulk_wait_read<0>();   // this warp's previous store has read its rows
          __syncwarp();
        }
        if (hsel == 0)
          finish_pair<0>(p, tmem_row, buf, zs2, stg, r);
        else
          finish_pair<1>(p, tmem_row, buf, zs2, stg, r);
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tempty[buf]);
          mbar_arrive(&sempty[sb]);
          // rows 32q .. 32q+31 of the box: one TMA store (pairs past the block's edge are clipped by
          // the map, whose extents are the block's)
          if (jt * BM + q * 32 < p.bj) {
            tma_store_3d(&omap, stg + q * 32 * 128, hsel * 64, jt * BM + q * 32, il);
            bulk_commit();
          }
          if (!X16) {
            bulk_wait_read<0>();
            mbar_arrive(hempty);
          }
        }
      }
      if (lane == 0) bulk_wait_all();   // stores out before the CTA's shared memory goes away
    }
  }

  __syncthreads();
  if (*abort_flag) {
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 2000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_finish_bf16(bool x16, const CUtensorMap& xmap, const CUtensorMap& zmap,
                               const CUtensorMap& womap, const CUtensorMap& wgmap, const CUtensorMap& omap,
                               const FinishParams& p, int num_sms, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k3_finish<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k3_finish<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.total_tiles <= 0) return cudaSuccess;
  const int grid = (int)(p.total_tiles < num_sms ? p.total_tiles : num_sms);
  if (x16)
    k3_finish<true><<<grid, THREADS, SMEM_BYTES, s>>>(xmap, zmap, womap, wgmap, omap, p);
  else
    k3_finish<false><<<grid, THREADS, SMEM_BYTES, s>>>(xmap, zmap, womap, wgmap, omap, p);
  return cudaGetLastError();
}

}  // namespace tmk
