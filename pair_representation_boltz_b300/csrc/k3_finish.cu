// k3_finish.cu -- output stage of the triangle multiplicative update on the
// sm_103a tensor cores, over one output block:
//
//   out_ij = sigmoid(W_g zh_ij) * W_o LayerNorm_out(x_ij),   zh = LayerNorm_in(z)
//
// x comes float32 channel-major [128][bi][ldx] from the contraction; z and out
// are the caller's bf16 [N][N][128] pair representation (the layer(x, mask)
// call of the code-sample section of "NVIDIA BioNeMo escala modelagem
// biomolecular com context parallelism e quebra barreira de memória da GPU").
//
// Per tile of 128 pairs (one row i, 128 consecutive j of the block):
//   warp 0      TMA: x tile [128 c][128 j] fp32 (64 KB), z tile (two 64-channel
//               boxes, 128-byte swizzle); W_o (fp16) and W_g (bf16 hi + lo) once.
//   warps 2..5  thread = pair. LayerNorm of x over its 128 channels in fp32,
//               written back as fp16 rows of a K-major operand; LayerNorm
//               statistics of z. Then, one tile later, the epilogue of the
//               previous tile from TMEM: gate, product, 16-byte stores of out.
//   warp 1      tcgen05.mma: D[p][0..128) = xh x W_o'^T (kind::f16, fp16),
//               D[p][128..256) = z x W_g'^T (bf16, hi and lo), two TMEM buffers.
// LayerNorm_out's gamma is folded into W_o' = W_o diag(gamma_out) (scaled by a
// power of two to use fp16's range) and beta into a bias; LayerNorm_in of the
// gate is folded as in the projection: W_g zh = rstd (W_g' z - mu rowsum) + bias.
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int BM = kFinishTileJ;             // pairs per tile
constexpr int X_BYTES = kC * BM * 4;         // 64 KB fp32 [c][j]
constexpr int XH_BYTES = BM * kC * 2;        // 32 KB fp16, two K-chunks
constexpr int Z_BYTES = BM * kC * 2;         // 32 KB bf16, two K-chunks
constexpr int WO_BYTES = kC * kC * 2;        // 32 KB fp16
constexpr int WG_BYTES = 2 * kC * kC * 2;    // 64 KB bf16 hi + lo
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = X_BYTES + XH_BYTES + Z_BYTES + WO_BYTES + WG_BYTES + 3 * kC * 4 + 256;
constexpr int TMEM_COLS = 512;

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(kBoxFinishX.bytes() == X_BYTES, "x tile = one box");
static_assert(2 * kBoxFinishZ.bytes() == Z_BYTES, "z tile = two boxes");
static_assert(2 * kBoxFinishW.bytes() == WO_BYTES && 4 * kBoxFinishW.bytes() == WG_BYTES, "weight boxes");

__global__ void __launch_bounds__(THREADS, 1)
    k3_finish(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap zmap,
              const __grid_constant__ CUtensorMap womap, const __grid_constant__ CUtensorMap wgmap,
              const FinishParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* zs = smem;                        // 1024-aligned swizzled tiles first
  uint8_t* xh = zs + Z_BYTES;
  uint8_t* wo = xh + XH_BYTES;
  uint8_t* wg = wo + WO_BYTES;               // hi chunks then lo chunks
  float* xs = reinterpret_cast<float*>(wg + WG_BYTES);
  float* cst = xs + kC * BM;                 // rowsum_g[128], bias_g[128], bias_o[128]
  uint64_t* xfull = reinterpret_cast<uint64_t*>(cst + 3 * kC);
  uint64_t* xempty = xfull + 1;
  uint64_t* zfull = xempty + 1;
  uint64_t* zempty = zfull + 1;
  uint64_t* hfull = zempty + 1;
  uint64_t* hempty = hfull + 1;
  uint64_t* tfull = hempty + 1;
  uint64_t* tempty = tfull + 2;
  uint64_t* wfull = tempty + 2;
  uint64_t* fin = wfull + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
    if (*abort_flag) raise_status(p.w, ST_TIMEOUT, 90);
    mbar_init(xfull, 1);
    mbar_init(xempty, 4);
    mbar_init(zfull, 1);
    mbar_init(zempty, 1);
    mbar_init(hfull, 4);
    mbar_init(hempty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(wfull, 1);
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (threadIdx.x >= 64)
    for (int t = threadIdx.x - 64; t < 3 * kC; t += THREADS - 64) cst[t] = p.consts[t];
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
      if (lane == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&zmap);
        mbar_expect_tx(wfull, WO_BYTES + WG_BYTES);
        for (int kc = 0; kc < 2; ++kc) tma_load_2d(wo + kc * (WO_BYTES / 2), &womap, wfull, kc * 64, 0);
        for (int hl = 0; hl < 2; ++hl)
          for (int kc = 0; kc < 2; ++kc)
            tma_load_2d(wg + (hl * 2 + kc) * (WO_BYTES / 2), &wgmap, wfull, kc * 64, hl * kC);
        uint32_t ph = 0;
        for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
          const int il = (int)(t / p.tiles_j);
          const int jt = (int)(t - (long long)il * p.tiles_j);
          if (!wait_bounded(xempty, ph ^ 1u, p.w, abort_flag, 31)) break;
          mbar_expect_tx(xfull, X_BYTES);
          tma_load_3d(xs, &xmap, xfull, jt * BM, il, 0);
          if (!wait_bounded(zempty, ph ^ 1u, p.w, abort_flag, 32)) break;
          mbar_expect_tx(zfull, Z_BYTES);
          tma_load_3d(zs, &zmap, zfull, 0, p.j0 + jt * BM, p.i0 + il);
          tma_load_3d(zs + Z_BYTES / 2, &zmap, zfull, 64, p.j0 + jt * BM, p.i0 + il);
          ph ^= 1u;
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t id_y = make_idesc(BM, kC, FMT_F16, false, false);
        constexpr uint32_t id_g = make_idesc(BM, kC, FMT_BF16, false, false);
        uint32_t ph = 0;
        int local = 0;
        if (wait_bounded(wfull, 0, p.w, abort_flag, 33)) {
          const uint32_t h0 = smem_u32(xh), z0 = smem_u32(zs), o0 = smem_u32(wo), g0 = smem_u32(wg);
          for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!wait_bounded(&tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 34)) break;
            if (!wait_bounded(hfull, ph, p.w, abort_flag, 35)) break;
            if (!wait_bounded(zfull, ph, p.w, abort_flag, 36)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(buf * 2 * kC);
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
            mma_commit(hempty);
            mma_commit(zempty);
            mma_commit(&tfull[buf]);
            ph ^= 1u;
          }
        }
        mma_commit(fin);
        wait_bounded(fin, 0, p.w, abort_flag, 37);
      }
    } else {
      // ------------------------------------------------------------ LayerNorm + epilogue, thread = pair
      const int q = warp & 3;
      const int r = q * 32 + lane;
      uint32_t ph = 0;
      int local = 0;
      // state of the previous tile, whose epilogue runs after this tile's LayerNorm
      float pmu = 0.f, prs = 0.f;
      int pi = -1, pj = 0;
      bool pvalid = false;
      bool ok = true;
      for (long long t = blockIdx.x;; t += gridDim.x, ++local) {
        const bool have = t < p.total_tiles;
        float zmu = 0.f, zrs = 0.f;
        int ci = 0, cj = 0;
        bool cvalid = false;
        if (have) {
          const int il = (int)(t / p.tiles_j);
          const int jt = (int)(t - (long long)il * p.tiles_j);
          ci = p.i0 + il;
          cj = p.j0 + jt * BM + r;
          cvalid = (jt * BM + r) < p.bj;
          // statistics of z_ij
          if (!warp_wait_bounded(zfull, ph, p.w, abort_flag, 38)) {
            ok = false;
            break;
          }
          {
            float v[kC];
#pragma unroll
            for (int kc = 0; kc < 2; ++kc)
#pragma unroll
              for (int uu = 0; uu < 8; ++uu) {
                const uint4 w4 = *reinterpret_cast<const uint4*>(zs + kc * (Z_BYTES / 2) + sw128_offset(r, uu));
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w4);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __bfloat1622float2(h[e]);
                  v[kc * 64 + uu * 8 + 2 * e] = f.x;
                  v[kc * 64 + uu * 8 + 2 * e + 1] = f.y;
                }
              }
            float s0 = 0.f;
#pragma unroll
            for (int c = 0; c < kC; ++c) s0 += v[c];
            zmu = s0 * (1.0f / kC);
            float s1 = 0.f;
#pragma unroll
            for (int c = 0; c < kC; ++c) s1 += (v[c] - zmu) * (v[c] - zmu);
            zrs = rsqrtf(s1 * (1.0f / kC) + 1e-5f);
          }
          // LayerNorm of x_ij over channels -> fp16 operand row
          if (!warp_wait_bounded(xfull, ph, p.w, abort_flag, 39)) {
            ok = false;
            break;
          }
          float v[kC];
#pragma unroll
          for (int c = 0; c < kC; ++c) v[c] = xs[c * BM + r];
          __syncwarp();
          if (lane == 0) mbar_arrive(xempty);
          float s0 = 0.f;
#pragma unroll
          for (int c = 0; c < kC; ++c) s0 += v[c];
          const float xmu = s0 * (1.0f / kC);
          float s1 = 0.f;
#pragma unroll
          for (int c = 0; c < kC; ++c) s1 += (v[c] - xmu) * (v[c] - xmu);
          const float xrs = rsqrtf(s1 * (1.0f / kC) + 1e-5f);
          if (!warp_wait_bounded(hempty, ph ^ 1u, p.w, abort_flag, 40)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int uu = 0; uu < 8; ++uu) {
              const int c = kc * 64 + uu * 8;
              uint4 w4;
              w4.x = pack_f16x2((v[c + 0] - xmu) * xrs, (v[c + 1] - xmu) * xrs);
              w4.y = pack_f16x2((v[c + 2] - xmu) * xrs, (v[c + 3] - xmu) * xrs);
              w4.z = pack_f16x2((v[c + 4] - xmu) * xrs, (v[c + 5] - xmu) * xrs);
              w4.w = pack_f16x2((v[c + 6] - xmu) * xrs, (v[c + 7] - xmu) * xrs);
              *reinterpret_cast<uint4*>(xh + kc * (XH_BYTES / 2) + sw128_offset(r, uu)) = w4;
            }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(hfull);
          ph ^= 1u;
        }
        // epilogue of the previous tile
        if (local > 0) {
          const int pl = local - 1;
          const int buf = pl & 1;
          const uint32_t use = (uint32_t)(pl >> 1);
          if (!warp_wait_bounded(&tfull[buf], use & 1u, p.w, abort_flag, 41)) {
            ok = false;
            break;
          }
          tc_fence_after();
          __nv_bfloat16* dst = p.out + ((size_t)pi * p.N + pj) * kC;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t yv[32], gv[32];
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 2 * kC + cc * 32);
            tmem_ld32(ta, yv);
            tmem_ld32(ta + kC, gv);
            tmem_ld_wait();
            if (pvalid) {
              uint32_t packed[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float o2[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int o = cc * 32 + e + h;
                  const float y = __uint_as_float(yv[e + h]) * p.inv_scale_o + cst[2 * kC + o];
                  const float g = prs * (__uint_as_float(gv[e + h]) - pmu * cst[o]) + cst[kC + o];
                  o2[h] = sigmoidf_fast(g) * y;
                }
                packed[e / 2] = pack_bf16x2(o2[0], o2[1]);
              }
              uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                d4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        if (!have) break;
        pmu = zmu;
        prs = zrs;
        pi = ci;
        pj = cj;
        pvalid = cvalid;
      }
      (void)ok;
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

cudaError_t launch_finish_bf16(const CUtensorMap& xmap, const CUtensorMap& zmap, const CUtensorMap& womap,
                               const CUtensorMap& wgmap, const FinishParams& p, int num_sms, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k3_finish, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.total_tiles <= 0) return cudaSuccess;
  const int grid = (int)(p.total_tiles < num_sms ? p.total_tiles : num_sms);
  k3_finish<<<grid, THREADS, SMEM_BYTES, s>>>(xmap, zmap, womap, wgmap, p);
  return cudaGetLastError();
}

}  // namespace tmk
