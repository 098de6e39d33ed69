// k2_contract.cu -- the per-channel contraction of the triangle multiplicative
// update on the sm_103a tensor cores.
//
//   outgoing: x_ij = sum_k a_ik b_jk   (X_c = A_c B_c^T)
//   incoming: x_ij = sum_k a_ki b_kj   (X_c = A_c^T B_c)
//
// a and b are channel-major bf16 [128][N][ld]; x is [128][bi][ldx] for one
// output block (i0, j0, bi, bj), float32 or fp16 scaled by one power of two
// chosen on the host so that no value can leave fp16's range. This is the O(N^3 c) step that the
// 2D block tiling of the pair representation exists for ("2D tiling da pair
// representation" section of "NVIDIA BioNeMo escala modelagem biomolecular com
// context parallelism e quebra barreira de memória da GPU"); here the N x N
// grid is tiled inside one GPU.
//
// Design: clusters of two CTAs (one per SM), persistent over (channel, i-tile,
// j-tile) with 256 x 256 output tiles (the last tile column only as wide as the
// columns it has left, rounded up to 16: a narrower MMA, not wasted work). The pair's tensor cores run one
// M = 256, N = 256 MMA: each CTA stages its own 128 rows of A and its own 128
// of the tile's 256 B rows, so that per multiply-add each SM reads half the B
// bytes a single-CTA 128 x 256 tile would need, from L2 and from shared memory.
//   warp 0      (both CTAs) TMA producer: 128 x 64 A and 128 x 64 B per stage,
//               128-byte swizzle, 6-stage ring; completion of both CTAs' copies
//               is counted on the first CTA's "full" barrier, the stage's
//               release arrives on both CTAs' "empty" barriers.
//   warp 1      TMEM (512 columns, two 256-column accumulators, allocated in both
//               CTAs together); in the first CTA, the single-thread issuer of
//               tcgen05.mma.cta_group::2 (K = 16 per instruction, f32 accumulate).
//   warps 2..5  (both CTAs) epilogue of the CTA's 128 rows: tcgen05.ld 32 columns
//               at a time into a per-warp 128-byte-swizzled staging tile (two per
//               warp), TMA store of each 32 x 32 float32 (or 32 x 64 fp16) sub-tile;
//               TMA clips the block edges. The accumulator goes back to the MMA issuer when the
//               warps of both CTAs have arrived on the first CTA's barrier.
//               (Blocks whose origin is not a multiple of 8 fall back to direct
//               16-byte stores: a TMA box must not start below zero or off its
//               16-byte inner-axis grid.)
// Incoming reads the same a/b buffers through tensor maps whose box runs along
// the other pair index ("transposed" boxes), and tells the MMA that A and B are
// M/N-major; no transpose is ever materialised. A third form, with A read as in
// the outgoing contraction and B as in the incoming one (x_ij = sum_k A_ik B_kj),
// serves the backward pass's products of dL/dx with a or b. k beyond N is
// zero-filled by TMA.
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int BM = kContractBM, BN = kContractBN, BK = kContractBK;   // 256 x 256 tile of the pair
constexpr int HM = BM / 2, HN = BN / 2;       // rows of A and of B staged by each CTA
constexpr int STAGES = 6;
constexpr int A_BYTES = HM * BK * 2;          // 16 KB
constexpr int B_BYTES = HN * BK * 2;          // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;             // two accumulators
constexpr int THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr int STG_BYTES = 32 * 32 * 4;        // one 32 x 32 float32 staging tile
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_WARPS * 2 * STG_BYTES + 256;

static_assert(TMEM_COLS == 512, "two 256-column accumulators fill TMEM");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(kBoxContractOutA.bytes() == A_BYTES && kBoxContractOutB.bytes() == B_BYTES, "outgoing boxes");
static_assert(2 * kBoxContractIn.bytes() == A_BYTES && 2 * kBoxContractIn.bytes() == B_BYTES, "incoming boxes");
static_assert(kBoxContractX.bytes() == STG_BYTES && kBoxContractX16.bytes() == STG_BYTES, "x store boxes");

struct Tile {
  int c, ti, tj;
};
__device__ __forceinline__ Tile decode(long long t, const ContractParams& p) {
  const long long per_c = (long long)p.tiles_i * p.tiles_j;
  Tile r;
  r.c = (int)(t / per_c);
  const int rem = (int)(t - (long long)r.c * per_c);
  r.ti = rem / p.tiles_j;
  r.tj = rem - r.ti * p.tiles_j;
  return r;
}

// MODE: the operands' forms (ContractMode); X16: x leaves as fp16 scaled by 2^x_exp, else float32.
template <int MODE, bool X16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k2_contract(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                const __grid_constant__ CUtensorMap xmap, const ContractParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  uint8_t* stg = smem + STAGES * STAGE_BYTES;     // [epilogue warp][2][32 x 32 float32], 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + EPI_WARPS * 2 * STG_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();        // 0: issues the MMAs; 1: its peer
  const long long pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;  // swizzled tiles need 1024-byte alignment
    if (*abort_flag) raise_status(p.w, ST_TIMEOUT, 90);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);     // first CTA: its producer's arrival + both CTAs' bytes
      mbar_init(&empty[s], 1);    // both CTAs: the stage's MMAs have read it
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);                 // both CTAs: the accumulator is complete
      mbar_init(&tempty[b], 2 * EPI_WARPS);    // first CTA: both CTAs' epilogues are done with it
    }
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&bmap);
  }
  if (warp == 1) {
    tmem_alloc_pair(tslot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tslot;
  const int KB = (p.N + BK - 1) / BK;
  // the first CTA's barriers, as cluster-window addresses (valid from either CTA)
  const uint32_t full0 = mapa_cluster(smem_u32(full), 0);
  const uint32_t tempty0 = mapa_cluster(smem_u32(tempty), 0);
  if (!*abort_flag) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      if (lane == 0) {
        int s = 0;
        uint32_t ph = 0;
        for (long long t = pair; t < p.total_tiles; t += npairs) {
          const Tile tl = decode(t, p);
          // ia, jb are multiples of 8: the incoming boxes start there along their inner axis. The last
          // tile column runs a narrower MMA (N = last_n), whose second half of B comes from the peer.
          const int ntile = tl.tj == p.tiles_j - 1 ? p.last_n : BN;
          const int ia = p.i_base + tl.ti * BM + (int)rank * HM;
          const int jb = p.j_base + tl.tj * BN + (int)rank * (ntile / 2);
          for (int kb = 0; kb < KB; ++kb) {
            if (!wait_bounded(&empty[s], ph ^ 1u, p.w, abort_flag, 1)) goto producer_done;
            uint8_t* sa = tiles + s * STAGE_BYTES;
            uint8_t* sb = sa + A_BYTES;
            // the first CTA's "full" barrier counts the bytes of both CTAs' copies
            const uint32_t fb = rank == 0 ? smem_u32(&full[s]) : full0 + (uint32_t)(s * 8);
            if (rank == 0) mbar_expect_tx_u32(fb, 2 * STAGE_BYTES);
            if (MODE != CONTRACT_IN) {
              // A_c[i][k] = a_ik: rows i, k contiguous (K-major)
              tma_load_3d_pair(sa, &amap, fb, kb * BK, ia, tl.c);
            } else {
              // a_ki: rows k, i contiguous; 64-wide slabs along i (M-major)
              tma_load_3d_pair(sa, &amap, fb, ia, kb * BK, tl.c);
              tma_load_3d_pair(sa + 8192, &amap, fb, ia + 64, kb * BK, tl.c);
            }
            if (MODE == CONTRACT_OUT) {
              // B_c[j][k] = b_jk: rows j, k contiguous (K-major)
              tma_load_3d_pair(sb, &bmap, fb, kb * BK, jb, tl.c);
            } else {
              // b_kj: rows k, j contiguous; 64-wide slabs along j (N-major)
              tma_load_3d_pair(sb, &bmap, fb, jb, kb * BK, tl.c);
              tma_load_3d_pair(sb + 8192, &bmap, fb, jb + 64, kb * BK, tl.c);
            }
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      producer_done:;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer (first CTA)
      if (lane == 0 && rank == 0) {
        // bf16 operands (the update's a and b) or fp16 ones (the backward pass's)
        const uint32_t fmt = p.ab_f16 ? FMT_F16 : FMT_BF16;
        constexpr bool A_MN = MODE == CONTRACT_IN, B_MN = MODE != CONTRACT_OUT;
        const uint32_t idesc_full = make_idesc(BM, BN, fmt, A_MN, B_MN);
        const uint32_t idesc_last = make_idesc(BM, p.last_n, fmt, A_MN, B_MN);
        // descriptors of stage 0's A and B tiles; an operand's descriptor is its tile's plus the byte
        // offset / 16 (the start-address field, shared memory below 256 KB): formed once, not per MMA
        const uint32_t t0 = smem_u32(tiles);
        const uint64_t da = A_MN ? make_sdesc_sw128(t0, 8192, 1024) : make_sdesc_sw128(t0, 16, 1024);
        const uint64_t db = B_MN ? make_sdesc_sw128(t0 + A_BYTES, 8192, 1024) : make_sdesc_sw128(t0 + A_BYTES, 16, 1024);
        constexpr uint32_t KS_A = (A_MN ? 2048 : 32) >> 4, KS_B = (B_MN ? 2048 : 32) >> 4;
        int s = 0;
        uint32_t ph = 0;
        int local = 0;
        for (long long t = pair; t < p.total_tiles; t += npairs, ++local) {
          const int buf = local & 1;
          const uint32_t use = (uint32_t)(local >> 1);
          if (!wait_bounded(&tempty[buf], (use & 1u) ^ 1u, p.w, abort_flag, 2)) break;
          tc_fence_after();
          const uint32_t d = tmem_base + (uint32_t)(buf * BN);
          const uint32_t idesc = decode(t, p).tj == p.tiles_j - 1 ? idesc_last : idesc_full;
          bool ok = true;
          for (int kb = 0; kb < KB; ++kb) {
            if (!wait_bounded(&full[s], ph, p.w, abort_flag, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t so = (uint32_t)s * (uint32_t)(STAGE_BYTES >> 4);
            const uint64_t ad = da + so, bd = db + so;
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              mma_f16_pair(d, ad + (uint32_t)(ks * KS_A), bd + (uint32_t)(ks * KS_B), idesc, (kb | ks) != 0);
            mma_commit_pair(&empty[s]);
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(&tfull[buf]);
        }
        // every MMA issued by this thread has completed before TMEM is released
        mma_commit_pair(fin);
        wait_bounded(fin, 0, p.w, abort_flag, 4);
      }
    } else {
      // ------------------------------------------------------------ epilogue (both CTAs)
      const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 belong to this warp
      const int r = q * 32 + lane;
      uint8_t* const my_stg = stg + (warp - 2) * 2 * STG_BYTES;
      int sb = 0;
      if (lane == 0 && p.tma_store) tma_prefetch_desc(&xmap);
      // fp16 x: every value times 2^x_exp, exact; |x| 2^x_exp <= 2^14 by the bound behind x_exp
      const float xs = X16 ? __int_as_float((127 + p.x_exp) << 23) : 1.f;
      // output columns per staged box: 32 float32 or 64 fp16 values (128-byte rows either way)
      constexpr int BOXW = X16 ? 64 : 32;
      int local = 0;
      for (long long t = pair; t < p.total_tiles; t += npairs, ++local) {
        const Tile tl = decode(t, p);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!warp_wait_bounded(&tfull[buf], use & 1u, p.w, abort_flag, 5)) break;
        tc_fence_after();
        const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
        if (p.tma_store) {
          // i_base == i0 and j_base == j0 here, so every coordinate is >= 0 and 32-aligned along j
          const int row0 = tl.ti * BM + (int)rank * HM + q * 32;
#pragma unroll 1
          for (int ch = 0; ch < BN / BOXW; ++ch) {
            const int col0 = tl.tj * BN + ch * BOXW;
            // Sub-tiles wholly outside the block are neither staged nor stored (warp-uniform). Every
            // staging write below is followed by exactly one committed store, which is what makes
            // "at most one group still reading" mean "the other buffer's store, not this one's".
            if (row0 >= p.bi || col0 >= p.bj) break;
            uint32_t v[32], w[32];
            tmem_ld32(trow + (uint32_t)(ch * BOXW), v);
            if (X16) tmem_ld32(trow + (uint32_t)(ch * BOXW + 32), w);
            tmem_ld_wait();
            uint8_t* sbuf = my_stg + sb * STG_BYTES;
            if (lane == 0) bulk_wait_read<1>();   // the store that last read this buffer is done with it
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              uint4 val;
              if (X16) {
                const uint32_t* src = u < 4 ? v + 8 * u : w + 8 * (u - 4);
                val = make_uint4(pack_f16x2(__uint_as_float(src[0]) * xs, __uint_as_float(src[1]) * xs),
                                 pack_f16x2(__uint_as_float(src[2]) * xs, __uint_as_float(src[3]) * xs),
                                 pack_f16x2(__uint_as_float(src[4]) * xs, __uint_as_float(src[5]) * xs),
                                 pack_f16x2(__uint_as_float(src[6]) * xs, __uint_as_float(src[7]) * xs));
              } else {
                val = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
              }
              *reinterpret_cast<uint4*>(sbuf + sw128_offset(lane, u)) = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (!X16 && p.accumulate) tma_reduce_add_3d(&xmap, sbuf, col0, row0, tl.c);   // x += product
              else tma_store_3d(&xmap, sbuf, col0, row0, tl.c);
              bulk_commit();
            }
            sb ^= 1;
          }
        } else {
          // block-local row of this thread's TMEM lane, and block-local column of the tile's first column
          const int il = p.i_base + tl.ti * BM + (int)rank * HM + r - p.i0;
          const bool row_ok = il >= 0 && il < p.bi;
          const int jl0 = p.j_base + tl.tj * BN - p.j0;   // in (-8, bj)
          const long long row_off = (long long)tl.c * p.chan_stride + (long long)(row_ok ? il : 0) * p.ldx;
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t v[32];
            tmem_ld32(trow + (uint32_t)(ch * 32), v);
            tmem_ld_wait();
            const int jc = jl0 + ch * 32;
            if (!row_ok || jc >= p.bj || jc + 32 <= 0) continue;
            if (X16) {
              __half* xrow = reinterpret_cast<__half*>(p.x) + row_off;
              if (jc >= 0 && jc + 32 <= p.bj && (jc & 7) == 0) {
                // 16-byte aligned: x, ldx and chan_stride are multiples of 8 halves
#pragma unroll
                for (int e = 0; e < 32; e += 8)
                  *reinterpret_cast<uint4*>(xrow + jc + e) = make_uint4(
                      pack_f16x2(__uint_as_float(v[e]) * xs, __uint_as_float(v[e + 1]) * xs),
                      pack_f16x2(__uint_as_float(v[e + 2]) * xs, __uint_as_float(v[e + 3]) * xs),
                      pack_f16x2(__uint_as_float(v[e + 4]) * xs, __uint_as_float(v[e + 5]) * xs),
                      pack_f16x2(__uint_as_float(v[e + 6]) * xs, __uint_as_float(v[e + 7]) * xs));
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (jc + e >= 0 && jc + e < p.bj) xrow[jc + e] = __float2half_rn(__uint_as_float(v[e]) * xs);
              }
            } else {
              float* xrow = reinterpret_cast<float*>(p.x) + row_off;
              if (jc >= 0 && jc + 32 <= p.bj && (jc & 3) == 0) {
                // 16-byte aligned: x, ldx and chan_stride are multiples of 4
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                  *reinterpret_cast<uint4*>(xrow + jc + e) = make_uint4(v[e], v[e + 1], v[e + 2], v[e + 3]);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (jc + e >= 0 && jc + e < p.bj) xrow[jc + e] = __uint_as_float(v[e]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(buf * 8));
      }
      if (lane == 0) bulk_wait_all();   // stores done before the CTA's shared memory goes away
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // give in-flight TMA copies (this CTA's and the peer's, which signal this CTA) time to land
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  cluster_sync_all();      // the peer's TMEM is written by the first CTA's MMAs: both are done first
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_contract_bf16(int mode, const CUtensorMap& amap, const CUtensorMap& bmap,
                                 const CUtensorMap& xmap, const ContractParams& p, int num_sms, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  cudaError_t err = once_per_device(attr_set, [] {
    const void* fns[5] = {(const void*)k2_contract<CONTRACT_OUT, false>, (const void*)k2_contract<CONTRACT_IN, false>,
                          (const void*)k2_contract<CONTRACT_OUT, true>, (const void*)k2_contract<CONTRACT_IN, true>,
                          (const void*)k2_contract<CONTRACT_MIXED, false>};
    for (const void* f : fns) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (err != cudaSuccess) return err;
  if (mode != CONTRACT_OUT && mode != CONTRACT_IN && mode != CONTRACT_MIXED) return cudaErrorInvalidValue;
  if (mode == CONTRACT_MIXED && p.x_f16) return cudaErrorInvalidValue;   // float32 x only (backward)
  if (p.total_tiles <= 0) return cudaSuccess;
  long long pairs = num_sms / 2;
  if (pairs > p.total_tiles) pairs = p.total_tiles;
  if (pairs < 1) pairs = 1;
  const int grid = (int)(2 * pairs);
  if (mode == CONTRACT_MIXED)
    k2_contract<CONTRACT_MIXED, false><<<grid, THREADS, SMEM_BYTES, s>>>(amap, bmap, xmap, p);
  else if (p.x_f16) {
    if (mode == CONTRACT_IN)
      k2_contract<CONTRACT_IN, true><<<grid, THREADS, SMEM_BYTES, s>>>(amap, bmap, xmap, p);
    else
      k2_contract<CONTRACT_OUT, true><<<grid, THREADS, SMEM_BYTES, s>>>(amap, bmap, xmap, p);
  } else {
    if (mode == CONTRACT_IN)
      k2_contract<CONTRACT_IN, false><<<grid, THREADS, SMEM_BYTES, s>>>(amap, bmap, xmap, p);
    else
      k2_contract<CONTRACT_OUT, false><<<grid, THREADS, SMEM_BYTES, s>>>(amap, bmap, xmap, p);
  }
  return cudaGetLastError();
}

}  // namespace tmk
