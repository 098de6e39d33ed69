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
// which keeps the weights accurate to ~2^-18; mu and rstd come from the same
// smem tile in fp32.
//
// One CTA per SM. CTA parity selects the half it computes (a: W_a | W_ga, or
// b: W_b | W_gb), so the two CTAs of a pair read each z tile once from HBM and
// once from L2. Per tile of 128 pairs (one row i, 128 consecutive j):
//   warp 0      TMA: z tile (two 64-channel boxes, 128-byte swizzle), 2 stages;
//               the hi and lo weights of the half once at start (128 KB).
//   warp 1      TMEM (2 x 256 columns) and tcgen05.mma with the channels on
//               the TMEM lanes: D_proj[c][p] = W'_proj z^T and D_gate[c][p] =
//               W'_gate z^T (M = 128 channels, N = 128 pairs), hi + lo each;
//               operand descriptors are formed once and offset per MMA (a
//               descriptor built per MMA doubles the thread's issue time).
//   warps 2..5  LayerNorm statistics, thread = pair: one pass over the z row
//               (sums of z - z_0 and of its square, fp32x2; the shift by the
//               row's first value keeps the variance free of cancellation for
//               rows whose mean is far from zero), the z tile released as soon
//               as it is read; one tile ahead of the epilogue, double-buffered
//               in shared memory behind mbarriers, with the pair mask as one
//               bit per pair (warp ballot).
//   warps 6..21 epilogue, thread = channel: four warps per TMEM lane quadrant
//               split the 128 pairs, 32 each (four epilogue warps per SMSP hide
//               each other's latency); per-channel folding constants live in
//               registers; two pairs at a time in fp32x2 arithmetic, the
//               two sigmoids with two exponentials and one shared reciprocal
//               (three MUFU operations), no branch. Results go through
//               shared memory: each warp fills its own 32-channel x 32-pair
//               staging box (64-byte swizzle) that its lane 0 writes out with
//               one TMA store per tile, so channel rows leave as 64-byte lines
//               and no warp waits for another; the store drains while the next
//               tile's MMA runs. Each 16-pair chunk of the warp's accumulator
//               columns is read by two TMEM loads (projection, gate) under one
//               wait, and the wait for the last store to have read the staging
//               box comes after the first chunk's arithmetic. (Stores straight
//               from the threads, one channel row per lane, scatter each warp
//               instruction over 32 DRAM pages and ran 6x slower.)
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int BM = kProjTileJ;                 // pairs per tile
constexpr int STAGES = 2;
constexpr int Z_BYTES = BM * kC * 2;           // 32 KB (two 16 KB K-chunks)
constexpr int W_MAT = kC * kC * 2;             // one 128 x 128 bf16 matrix, two K-chunks: 32 KB
constexpr int W_BYTES = 4 * W_MAT;             // proj hi, proj lo, gate hi, gate lo
constexpr int STAT_WARPS = 4, EPI_WARPS = 16;
constexpr int THREADS = 64 + 32 * (STAT_WARPS + EPI_WARPS);   // TMA, MMA, statistics, epilogue warps
constexpr int OUT_BYTES = EPI_WARPS * (int)kBoxProjOut.bytes();      // one staging box per epilogue warp
constexpr int STAT_BUF = (BM / 2) * 16 + 16;   // float4 {rstd_2k, rstd_2k+1, nmu_2k, nmu_2k+1} + 4 mask words
constexpr int SMEM_BYTES = STAGES * Z_BYTES + W_BYTES + OUT_BYTES + 2 * STAT_BUF + 256;
constexpr int TMEM_COLS = 512;

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(2 * kBoxProjZ.bytes() == Z_BYTES, "z tile = two boxes");
static_assert(2 * kBoxProjW.bytes() == W_MAT, "weight matrix = two boxes");
static_assert(kBoxProjOut.d0 * 2 == 64 && kBoxProjOut.d2 == 32, "a staging box is 32 channel rows of 64 bytes");
static_assert(OUT_BYTES == 32768, "staging budget");

// F16OUT: a and b leave as fp16, each value rounded to bf16 first (the storage the update defines)
// and multiplied by the power of two p.out_scale[half], an exact step that the fp16 form of a
// normal-range bf16 value keeps exactly: the backward pass's contractions take fp16 operands.
template <bool F16OUT>
__global__ void __launch_bounds__(THREADS, 1)
    k1_project(const __grid_constant__ CUtensorMap zmap, const __grid_constant__ CUtensorMap wmap,
               const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
               const ProjectParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* zs = smem;
  uint8_t* ws = smem + STAGES * Z_BYTES;                  // [proj hi, proj lo, gate hi, gate lo]
  uint8_t* ostg = ws + W_BYTES;                           // [epilogue warp][32 channels][128 B], swizzled
  uint8_t* sbase = ostg + OUT_BYTES;                      // [2][STAT_BUF]
  uint64_t* zfull = reinterpret_cast<uint64_t*>(sbase + 2 * STAT_BUF);
  uint64_t* zempty = zfull + STAGES;
  uint64_t* tfull = zempty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;
  uint64_t* sempty = sfull + 2;
  uint64_t* wfull = sempty + 2;
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
      mbar_init(&zempty[s], 1 + STAT_WARPS);  // MMA commit + the statistics warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EPI_WARPS);
      mbar_init(&sfull[b], STAT_WARPS);
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
        tma_prefetch_desc(&zmap);
        tma_prefetch_desc(&wmap);
        // weights: rows (half*2 + hl)*256 + {0: projection, 128: gate} of the [2][2][256][128] array
        mbar_expect_tx(wfull, W_BYTES);
        for (int m = 0; m < 4; ++m) {
          const int hl = m & 1, gate = m >> 1;
          for (int kc = 0; kc < 2; ++kc)
            tma_load_2d(ws + m * W_MAT + kc * (W_MAT / 2), &wmap, wfull, kc * 64, (half * 2 + hl) * 256 + gate * 128);
        }
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
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc(kC, BM, FMT_BF16, false, false);
        int s = 0;
        uint32_t ph = 0;
        int local = 0;
        if (wait_bounded(wfull, 0, p.w, abort_flag, 12)) {
          // descriptors of the weight tiles and of z stage 0; an operand's descriptor is its tile's plus
          // the byte offset / 16 (the start-address field, shared memory below 256 KB)
          const uint64_t dw = make_sdesc_sw128(smem_u32(ws), 16, 1024);
          const uint64_t dz = make_sdesc_sw128(smem_u32(zs), 16, 1024);
          for (long long u = cta; u < p.total_tiles; u += nctas, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!wait_bounded(&tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 13)) break;
            if (!wait_bounded(&zfull[s], ph, p.w, abort_flag, 14)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(buf * 2 * BM);
            const uint64_t dzs = dz + (uint32_t)(s * (Z_BYTES >> 4));
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                constexpr uint32_t kW = W_MAT >> 4;
                const uint32_t off = (uint32_t)(kc * (W_MAT / 2) + ks * 32) >> 4;
                const uint64_t bd = dzs + (uint32_t)((kc * (Z_BYTES / 2) + ks * 32) >> 4);
                const uint32_t acc = (kc | ks) != 0;
                mma_f16(d, dw + off, bd, idesc, acc);
                mma_f16(d, dw + (kW + off), bd, idesc, 1u);
                mma_f16(d + BM, dw + (2 * kW + off), bd, idesc, acc);
                mma_f16(d + BM, dw + (3 * kW + off), bd, idesc, 1u);
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
    } else if (warp < 2 + STAT_WARPS) {
      // ------------------------------------------------------------ statistics, thread = pair
      const int sw = warp - 2;
      const int t = sw * 32 + lane;
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      for (long long u = cta; u < p.total_tiles; u += nctas, ++local) {
        const int i = (int)(u / p.tiles_per_row);
        const int jt = (int)(u - (long long)i * p.tiles_per_row);
        const int sb = local & 1;
        const uint32_t sph = (uint32_t)(local >> 1) & 1u;
        if (!warp_wait_bounded(&zfull[s], ph, p.w, abort_flag, 16)) break;
        const uint8_t* zt = zs + s * Z_BYTES;
        // one pass over the row: sums of d = z - z_0 and of d^2 (fp32x2), shifted by the row's first
        // value; the z tile is released as soon as the row is in registers
        uint4 raw[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          raw[k] = *reinterpret_cast<const uint4*>(zt + (k >> 3) * (Z_BYTES / 2) + sw128_offset(t, k & 7));
        __syncwarp();
        if (lane == 0) mbar_arrive(&zempty[s]);     // this warp has finished reading the z tile
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
        const float z0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(&raw[0].x));
        const float2 nz0 = make_float2(-z0, -z0);
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float2 sq[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 d = __fadd2_rn(__bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e])), nz0);
            acc[e & 1] = __fadd2_rn(acc[e & 1], d);
            sq[e & 1] = __ffma2_rn(d, d, sq[e & 1]);
          }
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]);
        const float2 s01 = __fadd2_rn(sq[0], sq[1]);
        const float dm = (a01.x + a01.y) * (1.0f / kC);            // mean of d
        const float mu = z0 + dm;
        const float var = fmaxf((s01.x + s01.y) * (1.0f / kC) - dm * dm, 0.f);
        const float rstd = rsqrtf(var + 1e-5f);
        const int j = jt * BM + t;
        // the finish kernel's gate reads the same LayerNorm_in statistics (one CTA of the pair writes
        // them: 256 contiguous bytes per warp)
        if (p.zstat && half == 0 && j < p.N) p.zstat[(size_t)i * p.N + j] = make_float2(rstd, -rstd * mu);
        float m = 0.f;
        if (j < p.N) m = (p.mask ? p.mask[i] : 1.0f) * (p.mask_col ? p.mask_col[j] : 1.0f);
        const unsigned bits = __ballot_sync(0xffffffffu, m != 0.f);
        // the epilogue of two tiles ago has let go of this buffer
        if (!warp_wait_bounded(&sempty[sb], sph ^ 1u, p.w, abort_flag, 18)) break;
        float* st = reinterpret_cast<float*>(sbase + sb * STAT_BUF);
        st[(t >> 1) * 4 + (t & 1)] = rstd;
        st[(t >> 1) * 4 + 2 + (t & 1)] = -rstd * mu;
        if (lane == 0) reinterpret_cast<uint32_t*>(sbase + sb * STAT_BUF + (BM / 2) * 16)[sw] = bits;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[sb]);
      }
    } else {
      // ------------------------------------------------------------ epilogue, thread = channel
      const int ew = warp - 2 - STAT_WARPS;    // 0..15
      const int q = warp & 3;                  // TMEM lane quadrant: channels 32q .. 32q+31
      const int c = q * 32 + lane;
      const int pbase = (ew >> 2) * 32;        // this warp's 32 pair columns
      const CUtensorMap* omap = half ? &bmap : &amap;
      uint8_t* const box = ostg + ew * (int)kBoxProjOut.bytes();
      const float* cst = p.consts + half * 512;
      const float2 rsp = make_float2(cst[c], cst[c]), rsg = make_float2(cst[kC + c], cst[kC + c]);
      const float2 bp = make_float2(cst[256 + c], cst[256 + c]), bg = make_float2(cst[256 + kC + c], cst[256 + kC + c]);
      const float2 one2 = make_float2(1.f, 1.f);
      const float osc = p.out_scale[half];
      if (lane == 0) tma_prefetch_desc(omap);
      int local = 0;
      for (long long u = cta; u < p.total_tiles; u += nctas, ++local) {
        const int i = (int)(u / p.tiles_per_row);
        const int jt = (int)(u - (long long)i * p.tiles_per_row);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        const int sb = local & 1;
        const uint32_t sph = (uint32_t)(local >> 1) & 1u;
        if (!warp_wait_bounded(&sfull[sb], sph, p.w, abort_flag, 19)) break;
        if (!warp_wait_bounded(&tfull[buf], use & 1u, p.w, abort_flag, 17)) break;
        tc_fence_after();
        const float4* st = reinterpret_cast<const float4*>(sbase + sb * STAT_BUF);
        const uint32_t* mw = reinterpret_cast<const uint32_t*>(sbase + sb * STAT_BUF + (BM / 2) * 16);
        const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 2 * BM + pbase);
        // a, b of pairs p0+e and p0+e+1 for this channel (fp32x2: folded LayerNorm, gate, product)
        auto pair_values = [&](int p0, int e, const uint32_t* pr, const uint32_t* gt) -> float2 {
          const float4 sv = st[(p0 + e) >> 1];          // rstd and -rstd*mu of the two pairs
          const float2 r = make_float2(sv.x, sv.y), n = make_float2(sv.z, sv.w);
          const float2 pre = __ffma2_rn(r, make_float2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                                        __ffma2_rn(n, rsp, bp));
          const float2 gpre = __ffma2_rn(r, make_float2(__uint_as_float(gt[e]), __uint_as_float(gt[e + 1])),
                                         __ffma2_rn(n, rsg, bg));
          // sigmoid of both gates with one reciprocal: the gate rows carry -log2(e), so gpre is
          // -g log2 e and with d = 1 + 2^gpre, sigmoid(g0) = d1 / (d0 d1), sigmoid(g1) = d0 / (d0 d1).
          // The exponent is capped at 63 so that d0 d1 < 2^127 (a gate below -43 then reads 2^-63
          // instead of ~0).
          float e0, e1, rd;
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(fminf(gpre.x, 63.f)));
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(fminf(gpre.y, 63.f)));
          const float2 den = __fadd2_rn(make_float2(e0, e1), one2);
          asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rd) : "f"(den.x * den.y));
          return __fmul2_rn(__fmul2_rn(make_float2(den.y, den.x), pre), make_float2(rd, rd));
        };
        // bf16 a, b (or their fp16 form, scaled by a power of two, for the backward pass)
        auto pack = [&](float x, float y) -> uint32_t {
          if (!F16OUT) return pack_bf16x2(x, y);
          const float2 r2 = __bfloat1622float2(__floats2bfloat162_rn(x, y));
          return pack_f16x2(r2.x * osc, r2.y * osc);
        };
        // two 16-pair chunks, each read by two TMEM loads (projection, gate) under one wait
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pr[16], gt[16];
          tmem_ld16(ta + (uint32_t)(hh * 16), pr);
          tmem_ld16(ta + BM + (uint32_t)(hh * 16), gt);
          tmem_ld_wait();
          const int p0 = pbase + hh * 16;
          const uint32_t mword = mw[p0 >> 5] >> (p0 & 31);
          uint32_t packed[8];
          if ((mword & 0xFFFFu) == 0xFFFFu) {
            // all 16 pairs unmasked and inside the grid (warp-uniform): no per-element mask
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float2 v = pair_values(p0, e, pr, gt);
              packed[e >> 1] = pack(v.x, v.y);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float2 v = pair_values(p0, e, pr, gt);
              packed[e >> 1] = pack(((mword >> e) & 1u) ? v.x : 0.f, ((mword >> (e + 1)) & 1u) ? v.y : 0.f);
            }
          }
          if (hh == 0) {
            // the last tile's store has finished reading the staging box (waited for only now, after the
            // first chunk's arithmetic)
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
          // 32 bytes of this channel's 64-byte staging row: 16-byte units 2hh, 2hh+1
#pragma unroll
          for (int k = 0; k < 2; ++k)
            *reinterpret_cast<uint4*>(box + sw64_offset(lane, hh * 2 + k)) =
                make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
        }
        // the accumulator and the statistics buffer are free (every TMEM load has been waited for)
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tempty[buf]);
          mbar_arrive(&sempty[sb]);
          // pairs past N are clipped by TMA (whole 16-byte granules, inside the row padding of ld)
          if (jt * BM + pbase < p.N) {
            tma_store_3d(omap, box, jt * BM + pbase, i, q * 32);
            bulk_commit();
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

cudaError_t launch_project_bf16(const CUtensorMap& zmap, const CUtensorMap& wmap, const CUtensorMap& amap,
                                const CUtensorMap& bmap, const ProjectParams& p, int num_sms, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  cudaError_t e = once_per_device(attr_set, [] {
    cudaError_t r = cudaFuncSetAttribute(k1_project<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(k1_project<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return r;
  });
  if (e != cudaSuccess) return e;
  if (p.total_tiles <= 0) return cudaSuccess;
  long long pairs = num_sms / 2;
  if (pairs > p.total_tiles) pairs = p.total_tiles;
  if (pairs < 1) pairs = 1;
  if (p.out_f16)
    k1_project<true><<<(int)(2 * pairs), THREADS, SMEM_BYTES, s>>>(zmap, wmap, amap, bmap, p);
  else
    k1_project<false><<<(int)(2 * pairs), THREADS, SMEM_BYTES, s>>>(zmap, wmap, amap, bmap, p);
  return cudaGetLastError();
}

}  // namespace tmk
