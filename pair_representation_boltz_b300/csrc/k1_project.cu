// k1_project.cu -- input LayerNorm, the four projections, sigmoid gates and
// pair mask of the triangle multiplicative update, on the sm_103a tensor cores:
//
//   a_ij = sigmoid(W_ga zh_ij) * (W_a zh_ij) * m_i m_j,   zh = LayerNorm_in(z)
//   b_ij = sigmoid(W_gb zh_ij) * (W_b zh_ij) * m_i m_j
//
// written channel-major as bf16 a[c][i][j], b[c][i][j] (row stride ld), the
// layout the contraction reads. The pair representation z [N][N][128] bf16 is
// the input of every Pairformer pair update (the layer of the code-sample
// section of "NVIDIA BioNeMo escala modelagem biomolecular com context
// parallelism e quebra barreira de memória da GPU").
//
// LayerNorm is folded into the GEMM so that the tensor cores read the raw,
// exact bf16 z: with W' = W diag(gamma_in),
//   W zh = rstd * (W' z - mu * rowsum(W')) + W beta_in.
// W' is split into bf16 hi + lo parts (two MMAs into one fp32 accumulator),
// which keeps the weights accurate to ~2^-17; mu and rstd come from the same
// smem tile in fp32.
//
// One CTA per SM. CTA parity selects the half it computes (a: W_a | W_ga, or
// b: W_b | W_gb), so the two CTAs of a pair read each z tile once from HBM and
// once from L2. Per tile of 128 pairs (one row i, 128 consecutive j):
//   warp 0      TMA: z tile (two 64-channel boxes, 128-byte swizzle), 3 stages;
//               the 256 x 128 hi and lo weights once at start (128 KB).
//   warp 1      TMEM (2 x 256 columns) and tcgen05.mma: D[p][0..256) =
//               z_tile x [W'_proj | W'_gate]^T, M = 128, N = 256.
//   warps 2..5  thread = pair: LayerNorm statistics from the z tile, then the
//               gated, masked epilogue from TMEM; each channel row of a/b gets
//               64 contiguous bytes per warp store.
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int BM = kProjTileJ;                 // pairs per tile
constexpr int NOUT = 256;                      // outputs per half: projection 128 + gate 128
constexpr int STAGES = 3;
constexpr int Z_BYTES = BM * kC * 2;           // 32 KB (two 16 KB K-chunks)
constexpr int W_CHUNK = NOUT * 64 * 2;         // 32 KB: 256 rows x 64 channels
constexpr int W_BYTES = 4 * W_CHUNK;           // hi/lo x two K-chunks
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = STAGES * Z_BYTES + W_BYTES + 512 * 4 + 256;
constexpr int TMEM_COLS = 512;

static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__global__ void __launch_bounds__(THREADS, 1)
    k1_project(const __grid_constant__ CUtensorMap zmap, const __grid_constant__ CUtensorMap wmap,
               const ProjectParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* zs = smem;
  uint8_t* ws = smem + STAGES * Z_BYTES;
  float* cst = reinterpret_cast<float*>(ws + W_BYTES);  // rowsum[256], bias[256]
  uint64_t* zfull = reinterpret_cast<uint64_t*>(cst + 512);
  uint64_t* zempty = zfull + STAGES;
  uint64_t* tfull = zempty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* wfull = tempty + 2;
  uint64_t* fin = wfull + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1;
  const int cta = blockIdx.x >> 1;
  const int nctas = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
    if (*abort_flag) raise_status(p.w, ST_TIMEOUT, 90);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&zfull[s], 1);
      mbar_init(&zempty[s], 1 + 4);  // MMA commit + 4 epilogue warps (statistics read)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(wfull, 1);
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (threadIdx.x >= 64) {
    for (int t = threadIdx.x - 64; t < 512; t += THREADS - 64) cst[t] = p.consts[half * 512 + t];
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
      if (lane == 0) {
        tma_prefetch_desc(&zmap);
        tma_prefetch_desc(&wmap);
        mbar_expect_tx(wfull, W_BYTES);
        for (int hl = 0; hl < 2; ++hl)
          for (int kc = 0; kc < 2; ++kc)
            tma_load_2d(ws + (hl * 2 + kc) * W_CHUNK, &wmap, wfull, kc * 64, (half * 2 + hl) * NOUT);
        int s = 0;
        uint32_t ph = 0;
        for (long long u = cta; u < p.total_tiles; u += nctas) {
          const int i = (int)(u / p.tiles_per_row);
          const int jt = (int)(u - (long long)i * p.tiles_per_row);
          if (!wait_bounded(&zempty[s], ph ^ 1u, p.w, abort_flag, 11)) break;
          uint8_t* dst = zs + s * Z_BYTES;
          mbar_expect_tx(&zfull[s], Z_BYTES);
          tma_load_3d(dst, &zmap, &zfull[s], 0, jt * BM, i);
          tma_load_3d(dst + Z_BYTES / 2, &zmap, &zfull[s], 64, jt * BM, i);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc(BM, NOUT, FMT_BF16, false, false);
        int s = 0;
        uint32_t ph = 0;
        int local = 0;
        if (wait_bounded(wfull, 0, p.w, abort_flag, 12)) {
          const uint32_t w0 = smem_u32(ws);
          for (long long u = cta; u < p.total_tiles; u += nctas, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!wait_bounded(&tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 13)) break;
            if (!wait_bounded(&zfull[s], ph, p.w, abort_flag, 14)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(buf * NOUT);
            const uint32_t z0 = smem_u32(zs + s * Z_BYTES);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ad = make_sdesc_sw128(z0 + kc * (Z_BYTES / 2) + ks * 32, 16, 1024);
                const uint64_t bh = make_sdesc_sw128(w0 + (0 * 2 + kc) * W_CHUNK + ks * 32, 16, 1024);
                const uint64_t bl = make_sdesc_sw128(w0 + (1 * 2 + kc) * W_CHUNK + ks * 32, 16, 1024);
                mma_f16(d, ad, bh, idesc, (kc | ks) != 0);
                mma_f16(d, ad, bl, idesc, 1u);
              }
            }
            mma_commit(&zempty[s]);
            mma_commit(&tfull[buf]);
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        mma_commit(fin);
        wait_bounded(fin, 0, p.w, abort_flag, 15);
      }
    } else {
      // ------------------------------------------------------------ statistics + epilogue, thread = pair
      const int q = warp & 3;
      const int r = q * 32 + lane;
      __nv_bfloat16* const outp = half ? p.b : p.a;
      const size_t chan = (size_t)p.N * (size_t)p.ld;
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      for (long long u = cta; u < p.total_tiles; u += nctas, ++local) {
        const int i = (int)(u / p.tiles_per_row);
        const int jt = (int)(u - (long long)i * p.tiles_per_row);
        const int j = jt * BM + r;
        const bool valid = j < p.N;
        // LayerNorm statistics of z_ij over its 128 channels (fp32, two passes over registers)
        if (!warp_wait_bounded(&zfull[s], ph, p.w, abort_flag, 16)) break;
        const uint8_t* zt = zs + s * Z_BYTES;
        uint4 raw[16];
#pragma unroll
        for (int kc = 0; kc < 2; ++kc)
#pragma unroll
          for (int uu = 0; uu < 8; ++uu)
            raw[kc * 8 + uu] = *reinterpret_cast<const uint4*>(zt + kc * (Z_BYTES / 2) + sw128_offset(r, uu));
        __syncwarp();
        if (lane == 0) mbar_arrive(&zempty[s]);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            sum += f.x + f.y;
          }
        }
        const float mu = sum * (1.0f / kC);
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            ss += (f.x - mu) * (f.x - mu) + (f.y - mu) * (f.y - mu);
          }
        }
        const float rstd = rsqrtf(ss * (1.0f / kC) + 1e-5f);
        float m = 0.f;
        if (valid) m = p.mask ? p.mask[i] * p.mask[j] : 1.0f;

        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!warp_wait_bounded(&tfull[buf], use & 1u, p.w, abort_flag, 17)) break;
        tc_fence_after();
        __nv_bfloat16* dst = outp + (size_t)i * p.ld + j;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t pr[32], gt[32];
          const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NOUT + cc * 32);
          tmem_ld32(ta, pr);
          tmem_ld32(ta + 128, gt);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int c = cc * 32 + e;
              const float pre = rstd * (__uint_as_float(pr[e]) - mu * cst[c]) + cst[256 + c];
              const float gpre = rstd * (__uint_as_float(gt[e]) - mu * cst[128 + c]) + cst[384 + c];
              dst[(size_t)c * chan] = __float2bfloat16_rn(sigmoidf_fast(gpre) * pre * m);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
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

cudaError_t launch_project_bf16(const CUtensorMap& zmap, const CUtensorMap& wmap, const ProjectParams& p,
                                int num_sms, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k1_project, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.total_tiles <= 0) return cudaSuccess;
  long long pairs = num_sms / 2;
  if (pairs > p.total_tiles) pairs = p.total_tiles;
  if (pairs < 1) pairs = 1;
  k1_project<<<(int)(2 * pairs), THREADS, SMEM_BYTES, s>>>(zmap, wmap, p);
  return cudaGetLastError();
}

}  // namespace tmk
