// k_backward.cu -- tensor-core (tcgen05) kernels of the bf16 backward pass, c_z = c_h = 128.
//
// The backward pass of the triangle multiplicative update (the layer of the code-sample section of
// "NVIDIA BioNeMo escala modelagem biomolecular com context parallelism e quebra barreira de
// memória da GPU", trained at larger crops as that page's section "A pegadinha" asks) is the chain
// rule through its steps in reverse. Two per-pair stages bracket the contraction gradients:
//
//   output backward (k_bwd_output), per pair p = (i, j):
//     zh = LN_in(z), xh = LN_out(x);  gg = W_g zh, y = W_o xh            [MMA 1: A = zh, xh]
//     dy = dout sigmoid(gg),  dgg = dout y sigmoid'(gg)
//     dxh = W_o^T dy,  dzh_g = W_g^T dgg                                  [MMA 2: A = dy, dgg]
//     dW_g += dgg zh^T,  dW_o += dy xh^T   (summed over the CTA's pairs)   [MMA 3, TMEM-resident]
//     dx = LN_out backward of dxh -> dX (fp16, times the power of two of a bound), d(gamma_out), d(beta_out)
//   projection backward (k_bwd_project), per pair p = (i, k), once for a and once for b:
//     pv = W_v zh, pg = W_gt zh                                            [MMA 1: A = zh]
//     dpv = dV sigmoid(pg) m_i m_k,  dpg = dV pv m_i m_k sigmoid'(pg)     (dV = dA or dB)
//     dzh += W_v^T dpv + W_gt^T dpg                                       [MMA 2, two accumulators]
//     dW_v += dpv zh^T,  dW_gt += dpg zh^T                                [MMA 3, TMEM-resident]
//     second launch: dz = LN_in backward of dzh, d(gamma_in), d(beta_in)
//
// Precision. Every tensor-core operand is fp16 (11 significant bits; bf16's 8 would cost several
// times the bf16 tolerance of the gradients), each stored times a power of two that keeps it inside
// fp16's normal range: the weight images and zh, xh by factors the weights fix (host), dy and dgg by
// factors from the largest |dout| (k_absmax_bf16, read here from device memory), the per-pair dpv and
// dpg by factors that bound them from the fp16 contraction operands. Every product's epilogue
// multiplies its float32 result by the exact inverse of the scales it carries, so all stored
// gradients (dzh, the parameter partials) are in true units. dX leaves as fp16 times the power of two
// that brings a bound on |dX| to 2^14: with r_x = 1/sqrt(var + eps) <= 1/sqrt(eps), |x_hat| <= sqrt(c),
// |dX_c| <= r_x (2 + sqrt(c)) max_c |gamma_out,c dxh_c| and |dxh_c| <= ||W_o[:, c]||_1 max |dout|, so the
// bound is a host constant times the largest |dout| (the same for every block of a block schedule).
//
// Blocks. The output backward runs over one block of the pair grid at a time (x of that block from the
// contraction), the projection backward over a range of whole grid rows; per-CTA partial sums are
// added to, so that a schedule of launches sums them (the host clears them first).
//
// Layout. One CTA of 512 threads per SM, persistent over tiles of 128 consecutive pairs of the
// flattened N x N grid. Warp w serves the 32 pairs of TMEM lane quarter w % 4 (the lanes it may
// read) and channel quarter w / 4: each pair is handled by four threads of 32 channels each, so
// that every warp's loads of a channel cover 32 consecutive pairs, and the LayerNorm statistics of a
// pair are combined from its four quarters through shared memory. Per-pair operands are written
// into 128 x 128 fp16 shared-memory tiles in the 128-byte-swizzled K-major layout (pair rows,
// channel columns). The same bytes serve MMA 1 and 2 as K-major operands (K =
// channels) and MMA 3 as MN-major operands (K = pairs): a 128-byte row of 64 channels of one pair is
// one K-major row and, read the other way, one MN-major row of 64 M (or N) elements at one K index.
// Weights are fp16 [out][in] images in the same layout; MMA 1 reads them K-major (B = W,
// N = out), MMA 2 MN-major (B = W^T, N = in, K = out). TMEM: columns 0..255 hold MMA 1's two
// results and then MMA 2's; columns 256..511 accumulate the two parameter gradients of MMA 3 over
// every tile of the CTA, written out once as per-CTA partial sums (added in fixed order later).
#include "pair_tile.cuh"

namespace tmk {
namespace {

using namespace pt;

struct alignas(1024) OutSmem {
  uint8_t zh[TILE], xh[TILE], dy[TILE], dgg[TILE], wg[TILE], wo[TILE];
  float ln[4 * kC];                     // gamma_in, beta_in, gamma_out, beta_out
  float red[4][2 * kC];                 // channel sums of each lane quarter, reduced at the end
  float2 xst[4][BT];                    // per channel quarter and pair: (mean, M2) of x
  float2 sst[4][BT];                    // per channel quarter and pair: sums of the LayerNorm backward
  uint64_t bar;
  uint32_t tmem_slot;
  int abort_flag;
};

struct alignas(1024) ProjSmem {
  uint8_t zh[TILE], dv[TILE], dg[TILE], wv[TILE], wgt[TILE];
  float ln[2 * kC];                     // gamma_in, beta_in
  float red[4][2 * kC];
  float2 sst[4][BT];
  uint64_t bar;
  uint32_t tmem_slot;
  int abort_flag;
};

// L2 prefetch of bytes [b0, b1) of a buffer, widened to 16-byte bounds (the caller keeps the
// widened range inside the buffer's allocation).
__device__ __forceinline__ void prefetch_range(const void* base, long long b0, long long b1) {
  const long long a0 = b0 & ~15ll, a1 = (b1 + 15) & ~15ll;
  if (a1 > a0) prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(base) + a0, (uint32_t)(a1 - a0));
}

// Prefetch, for the pairs [p0, p1) of a tile (N >= 128: at most two grid rows), channel c of a float32
// plane [128][N][ld] whose rows are 16-byte multiples.
__device__ __forceinline__ void prefetch_plane_rows(const float* plane, long long ld, int N, long long p0,
                                                    long long p1) {
  const int i = (int)(p0 / N), j0 = (int)(p0 - (long long)i * N);
  const int n1 = (int)((p1 - p0) < (long long)(N - j0) ? (p1 - p0) : (long long)(N - j0));
  prefetch_range(plane + (long long)i * ld, 4ll * j0, 4ll * (j0 + n1));
  if (p0 + n1 < p1) prefetch_range(plane + (long long)(i + 1) * ld, 0, 4ll * (p1 - p0 - n1));
}

}  // namespace


namespace {

// The 32 channels [32 h, 32 h + 32) of zh (times sz) for pair `pr` (LayerNorm_in from the stored
// statistics) into row r of an fp16 operand tile; zeros for a pair past the grid.
__device__ __forceinline__ void zh_quarter(uint8_t* tile, const float* ln_g, const float* ln_b, float sz,
                                           const __nv_bfloat16* z, const float2* zstat, long long pr, bool valid,
                                           int r, int h) {
  float f[32];
  if (valid) {
    const float2 st = zstat[pr];
    load32_bf16(z + pr * kC + 32 * h, f);
#pragma unroll
    for (int e = 0; e < 32; ++e) f[e] = (ln_g[32 * h + e] * fmaf(f[e], st.x, st.y) + ln_b[32 * h + e]) * sz;
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) f[e] = 0.f;
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) put8h(tile, r, 32 * h + 8 * u, f + 8 * u);
}

__global__ void __launch_bounds__(NT, 1) k_bwd_output(const BwdOutParams p) {
  extern __shared__ uint8_t smem_raw[];
  OutSmem& sm = *reinterpret_cast<OutSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lq = warp & 3, h = warp >> 2;          // TMEM lane quarter, channel quarter
  const int r = 32 * lq + lane;                    // pair row of the tile
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  for (int k = tid; k < 4 * kC; k += NT) sm.ln[k] = p.ln[k];
  copy_tile(sm.wg, p.w_g);
  copy_tile(sm.wo, p.w_o);
  if (warp == 0) {
    tmem_alloc(&sm.tmem_slot, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)(32 * lq) << 16);
  const float *g_in = sm.ln, *b_in = sm.ln + kC, *g_out = sm.ln + 2 * kC, *b_out = sm.ln + 3 * kC;
  const uint32_t a_zh = smem_u32(sm.zh), a_xh = smem_u32(sm.xh), a_dy = smem_u32(sm.dy), a_dgg = smem_u32(sm.dgg);
  const uint32_t a_wg = smem_u32(sm.wg), a_wo = smem_u32(sm.wo);
  const int c0 = 32 * h;                           // this thread's first channel
  // dy and dgg are stored times d1 and d2: powers of two that bring the largest |dout| to just below
  // 2^14, and its product with the bound on |y| / 4 likewise
  const float dmax = __uint_as_float(p.amax[0]);
  const float d1 = pow2_scale(dmax, 14), d2 = pow2_scale(dmax * p.y_bound4, 14);
  const float u_dxh = p.u_dxh / d1, u_dzh = p.u_dzh / d2, u_wg = p.u_wg / d2, u_wo = p.u_wo / d1;
  // dX's fp16 scale, from its bound; the projection backward reads the bound back from amax[1]
  const float dxb = p.dx_bound * dmax;
  const float sdx = pow2_scale(dxb, 14);
  if (blockIdx.x == 0 && tid == 0) p.amax[1] = __float_as_uint(dxb);

  float acc_g = 0.f, acc_b = 0.f;                  // channel c0 + lane: sums of dxh n and dxh
  float dx_max = 0.f;                              // largest |dX| this thread writes
  const long long PB = (long long)p.bi * p.bj;     // pairs of the block
  uint32_t phase = 0;
  int local = 0;
  bool ok = true;
  for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x, ++local) {
    const long long pl = t * BT + r;               // pair of the block
    const bool valid = pl < PB;
    const int il = valid ? (int)(pl / p.bj) : 0;
    const int jl = valid ? (int)(pl - (long long)il * p.bj) : 0;
    const int i = p.i0 + il, j = p.j0 + jl;
    const long long pr = (long long)i * p.N + j;   // pair of the grid
    const float* xp = p.x + (long long)il * p.ldx + jl + (long long)c0 * p.xplane;

    // ---- zh; x of this quarter (the contraction's output times x_unscale): (mean, M2), combined over
    // the four quarters (Chan et al.)
    zh_quarter(sm.zh, g_in, b_in, p.sz, p.z, p.zstat, pr, valid, r, h);
    float xv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) xv[e] = valid ? xp[e * p.xplane] * p.x_unscale : 0.f;
    {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) s += xv[e];
      const float m = s * (1.f / 32);
      float m2 = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) m2 = fmaf(xv[e] - m, xv[e] - m, m2);
      sm.xst[h][r] = make_float2(m, m2);
    }
    __syncthreads();
    float mu, rx;
    {
      const float2 q0 = sm.xst[0][r], q1 = sm.xst[1][r], q2 = sm.xst[2][r], q3 = sm.xst[3][r];
      mu = ((q0.x + q1.x) + (q2.x + q3.x)) * 0.25f;
      const float d0 = q0.x - mu, dd1 = q1.x - mu, dd2 = q2.x - mu, d3 = q3.x - mu;
      const float m2 = ((q0.y + q1.y) + (q2.y + q3.y)) + 32.f * ((d0 * d0 + dd1 * dd1) + (dd2 * dd2 + d3 * d3));
      rx = rsqrtf(m2 * (1.f / kC) + 1e-5f);
    }
    {
      float f[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = valid ? (g_out[c0 + e] * ((xv[e] - mu) * rx) + b_out[c0 + e]) * p.sx : 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) put8h(sm.xh, r, c0 + 8 * u, f + 8 * u);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma_tile(tmem, a_zh, false, a_wg, false, ID_KK_H, false);         // gg = W_g zh
      mma_tile(tmem + kC, a_xh, false, a_wo, false, ID_KK_H, false);    // y  = W_o xh
      mma_commit(&sm.bar);
    }
    if (!cta_wait(&sm.bar, phase, p.w, &sm.abort_flag, 1)) { ok = false; break; }
    phase ^= 1u;
    tc_fence_after();

    // ---- dy = dout g, dgg = dout y g (1 - g), channels [c0, c0 + 32), in two halves of 16
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t rg[16], ry[16];
      tmem_ld16(trow + c0 + 16 * hh, rg);
      tmem_ld16(trow + kC + c0 + 16 * hh, ry);
      float d[16];
      if (valid) {
        const uint4* q = reinterpret_cast<const uint4*>(p.dout + pr * kC + c0 + 16 * hh);
        const uint4 q0 = q[0], q1 = q[1];
        bf16x8_to_float(q0, d);
        bf16x8_to_float(q1, d + 8);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) d[e] = 0.f;
      }
      tmem_ld_wait();
      float vy[16], vg[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float s = sigmoid_mufu(__uint_as_float(rg[e]) * p.u_gg);
        vy[e] = d[e] * s * d1;
        vg[e] = d[e] * (__uint_as_float(ry[e]) * p.u_y) * s * (1.f - s) * d2;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        put8h(sm.dy, r, c0 + 16 * hh + 8 * u, vy + 8 * u);
        put8h(sm.dgg, r, c0 + 16 * hh + 8 * u, vg + 8 * u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma_tile(tmem, a_dy, false, a_wo, true, ID_KM_H, false);              // dxh   = W_o^T dy
      mma_tile(tmem + kC, a_dgg, false, a_wg, true, ID_KM_H, false);        // dzh_g = W_g^T dgg
      mma_tile(tmem + 2 * kC, a_dgg, true, a_zh, true, ID_MM_H, local > 0); // dW_g += dgg zh^T
      mma_tile(tmem + 3 * kC, a_dy, true, a_xh, true, ID_MM_H, local > 0);  // dW_o += dy xh^T
      mma_commit(&sm.bar);
    }
    {
      // L2 prefetch of what the next tile of this CTA reads: x (one channel per thread of the first
      // 128) and, for whole grid rows, z, dout and the LayerNorm_in statistics; issued here, where the
      // warps wait for the second MMA group anyway (one bulk request per lane takes the issuing warps
      // thousands of cycles)
      const long long tn = t + gridDim.x;
      if (tn < p.tiles && p.bj >= BT) {
        const long long q0 = tn * BT, q1 = (q0 + BT < PB) ? q0 + BT : PB;
        const long long g0 = (long long)p.i0 * p.N + q0, g1 = (long long)p.i0 * p.N + q1;
        if (tid < kC) prefetch_plane_rows(p.x + (long long)tid * p.xplane, p.ldx, p.bj, q0, q1);
        else if (p.bj == p.N && tid == kC) prefetch_range(p.z, g0 * 2 * kC, g1 * 2 * kC);
        else if (p.bj == p.N && tid == kC + 1) prefetch_range(p.dout, g0 * 2 * kC, g1 * 2 * kC);
        else if (p.bj == p.N && tid == kC + 2) prefetch_range(p.zstat, g0 * 8, g1 * 8);
      }
    }
    if (!cta_wait(&sm.bar, phase, p.w, &sm.abort_flag, 2)) { ok = false; break; }
    phase ^= 1u;
    tc_fence_after();

    // ---- dzh_g out; LayerNorm_out backward of dxh -> dX
    {
      uint32_t rz[32];
      tmem_ld32(trow + kC + c0, rz);
      tmem_ld_wait();
      if (valid && p.dzh)
#pragma unroll
        for (int e = 0; e < 32; ++e) p.dzh[(long long)(c0 + e) * p.dzh_P + (pr - p.dzh_off)] = __uint_as_float(rz[e]) * u_dzh;
    }
    uint32_t rd[32];
    tmem_ld32(trow + c0, rd);
    tmem_ld_wait();
    float s1 = 0.f, s2 = 0.f;
    {
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        xv[e] = valid ? (xv[e] - mu) * rx : 0.f;                  // n, the normalised x
        const float dxh = valid ? __uint_as_float(rd[e]) * u_dxh : 0.f;
        rd[e] = __float_as_uint(dxh);
        const float dn = dxh * g_out[c0 + e];
        s1 += dn;
        s2 = fmaf(dn, xv[e], s2);
        v[e] = dxh * xv[e];
      }
      acc_g += reduce_scatter32(v, lane);
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rd[e]);
      acc_b += reduce_scatter32(v, lane);
    }
    sm.sst[h][r] = make_float2(s1, s2);
    __syncthreads();
    {
      const float2 q0 = sm.sst[0][r], q1 = sm.sst[1][r], q2 = sm.sst[2][r], q3 = sm.sst[3][r];
      s1 = ((q0.x + q1.x) + (q2.x + q3.x)) * (1.f / kC);
      s2 = ((q0.y + q1.y) + (q2.y + q3.y)) * (1.f / kC);
    }
    if (valid && p.dx16) {
      __half* dp = p.dx16 + (long long)c0 * p.dxplane + (long long)i * p.ldd + j;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float dx = rx * (__uint_as_float(rd[e]) * g_out[c0 + e] - s1 - xv[e] * s2);
        dx_max = fmaxf(dx_max, fabsf(dx));
        dp[e * p.dxplane] = __float2half_rn(dx * sdx);
      }
    }
  }

  // ---- the largest |dX| written (the projection backward's scales of dpv, dpg follow from it)
  if (p.dx16) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dx_max = fmaxf(dx_max, __shfl_xor_sync(0xffffffffu, dx_max, o));
    if (lane == 0) atomicMax(p.amax + 2, __float_as_uint(dx_max));   // non-negative: bits order like values
  }

  // ---- per-CTA partial sums, added to: d(gamma_out), d(beta_out) over the lane quarters; dW_g, dW_o
  // from TMEM
  if (ok && p.part_w && local > 0) {
    sm.red[lq][c0 + lane] = acc_g;
    sm.red[lq][kC + c0 + lane] = acc_b;
    __syncthreads();
    for (int k = tid; k < 2 * kC; k += NT)
      p.part_ln[(long long)blockIdx.x * 2 * kC + k] += ((sm.red[0][k] + sm.red[1][k]) + sm.red[2][k]) + sm.red[3][k];
    float* pw = p.part_w + (long long)blockIdx.x * 2 * kC * kC + (long long)r * kC + c0;
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
      uint32_t rr[32];
      tmem_ld32(trow + (2 + m) * kC + c0, rr);
      tmem_ld_wait();
      const float u = m == 0 ? u_wg : u_wo;
#pragma unroll
      for (int e = 0; e < 32; ++e) pw[m * kC * kC + e] += __uint_as_float(rr[e]) * u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

namespace {

__global__ void __launch_bounds__(NT, 1) k_bwd_project(const BwdProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  ProjSmem& sm = *reinterpret_cast<ProjSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lq = warp & 3, h = warp >> 2;
  const int r = 32 * lq + lane;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  for (int k = tid; k < 2 * kC; k += NT) sm.ln[k] = p.ln[k];
  copy_tile(sm.wv, p.w_v);
  copy_tile(sm.wgt, p.w_gt);
  if (warp == 0) {
    tmem_alloc(&sm.tmem_slot, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)(32 * lq) << 16);
  const float *g_in = sm.ln, *b_in = sm.ln + kC;
  const uint32_t a_zh = smem_u32(sm.zh), a_dv = smem_u32(sm.dv), a_dg = smem_u32(sm.dg);
  const uint32_t a_wv = smem_u32(sm.wv), a_wgt = smem_u32(sm.wgt);
  const int c0 = 32 * h;
  // dV arrives times the fp16 scale of dX (from the bound in amax[1]) and times the fp16 scale of its
  // contraction partner (in the host factors below)
  // dpv, dpg are stored times q1, q2: powers of two from the largest |dV| the operands allow (N times
  // the largest fp16 dX, times the partner's 2^14), which keep them below 2^14 in fp16
  const float sdx = pow2_scale(__uint_as_float(p.amax[1]), 14);
  const float raw = p.q_raw * __uint_as_float(p.amax[2]) * sdx;
  const float q1 = pow2_scale(raw, 14), q2 = pow2_scale(raw * p.q2f, 14);
  const float u1 = p.u_dzh_v / (q1 * sdx), u2 = p.u_dzh_g / (q2 * sdx), u3 = p.u_wv / (q1 * sdx),
              u4 = p.u_wgt / (q2 * sdx);

  float acc_g = 0.f, acc_b = 0.f;
  uint32_t phase = 0;
  int local = 0;
  bool ok = true;
  for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x, ++local) {
    const long long pl = t * BT + r;               // pair of the range
    const bool valid = pl < p.P;
    const long long pr = p.p0 + (valid ? pl : 0);  // pair of the grid
    const int i = (int)(pr / p.N);
    const int k2 = (int)(pr - (long long)i * p.N);
    const long long hz = pr - p.dzh_off;           // its dzh column
    {
      // L2 prefetch of the next tile's dV (threads 0..127), dzh (128..255), z and statistics
      const long long tn = t + gridDim.x;
      if (tn < p.tiles && p.N >= BT) {
        const long long q0 = tn * BT, q1 = (q0 + BT < p.P) ? q0 + BT : p.P;
        const long long g0 = p.p0 + q0, g1 = p.p0 + q1, h0 = g0 - p.dzh_off, h1 = g1 - p.dzh_off;
        if (tid < kC) prefetch_plane_rows(p.dV + (long long)tid * p.vplane, p.ldv, p.N, q0, q1);
        else if (tid < 2 * kC) prefetch_range(p.dzh, ((tid - kC) * p.dzh_P + h0) * 4, ((tid - kC) * p.dzh_P + h1) * 4);
        else if (tid == 2 * kC) prefetch_range(p.z, g0 * 2 * kC, g1 * 2 * kC);
        else if (tid == 2 * kC + 1) prefetch_range(p.zstat, g0 * 8, g1 * 8);
      }
    }

    zh_quarter(sm.zh, g_in, b_in, p.sz, p.z, p.zstat, pr, valid, r, h);
    // this quarter of dV (issued before the MMA, consumed after it)
    const float m = valid ? (p.mask ? p.mask[i] * p.mask[k2] : 1.f) : 0.f;
    float dv[32];
    {
      const float* vp = p.dV + (long long)(i - p.i_off) * p.ldv + k2 + (long long)c0 * p.vplane;
#pragma unroll
      for (int e = 0; e < 32; ++e) dv[e] = valid ? vp[e * p.vplane] * m : 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma_tile(tmem, a_zh, false, a_wv, false, ID_KK_H, false);        // pv = W_v zh
      mma_tile(tmem + kC, a_zh, false, a_wgt, false, ID_KK_H, false);  // pg = W_gt zh
      mma_commit(&sm.bar);
    }
    if (!cta_wait(&sm.bar, phase, p.w, &sm.abort_flag, 1)) { ok = false; break; }
    phase ^= 1u;
    tc_fence_after();

    // ---- gate backward: dpv = dV s m, dpg = dV pv m s (1 - s), stored times q1, q2 (with dV's scale)
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t rv[16], rg[16];
      tmem_ld16(trow + c0 + 16 * hh, rv);
      tmem_ld16(trow + kC + c0 + 16 * hh, rg);
      tmem_ld_wait();
      float fv[16], fg[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float d = dv[16 * hh + e];
        const float s = sigmoid_mufu(__uint_as_float(rg[e]) * p.u_pg);
        fv[e] = d * s * q1;
        fg[e] = d * (__uint_as_float(rv[e]) * p.u_pv) * s * (1.f - s) * q2;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        put8h(sm.dv, r, c0 + 16 * hh + 8 * u, fv + 8 * u);
        put8h(sm.dg, r, c0 + 16 * hh + 8 * u, fg + 8 * u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      // the two terms of dzh carry different scales: one accumulator each
      mma_tile(tmem, a_dv, false, a_wv, true, ID_KM_H, false);               // W_v^T dpv
      mma_tile(tmem + kC, a_dg, false, a_wgt, true, ID_KM_H, false);         // W_gt^T dpg
      mma_tile(tmem + 2 * kC, a_dv, true, a_zh, true, ID_MM_H, local > 0);   // dW_v  += dpv zh^T
      mma_tile(tmem + 3 * kC, a_dg, true, a_zh, true, ID_MM_H, local > 0);   // dW_gt += dpg zh^T
      mma_commit(&sm.bar);
    }
    // the earlier terms of dzh, read while the MMA runs
    float dzh[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) dzh[e] = valid ? p.dzh[(long long)(c0 + e) * p.dzh_P + hz] : 0.f;
    if (!cta_wait(&sm.bar, phase, p.w, &sm.abort_flag, 2)) { ok = false; break; }
    phase ^= 1u;
    tc_fence_after();
    {
      uint32_t ra[32], rb[32];
      tmem_ld32(trow + c0, ra);
      tmem_ld32(trow + kC + c0, rb);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        dzh[e] = valid ? dzh[e] + (__uint_as_float(ra[e]) * u1 + __uint_as_float(rb[e]) * u2) : 0.f;
    }
    if (!p.final_pass) {
      if (valid)
#pragma unroll
        for (int e = 0; e < 32; ++e) p.dzh[(long long)(c0 + e) * p.dzh_P + hz] = dzh[e];
    } else {
      // LayerNorm_in backward: n = z rstd - rstd mu from the stored statistics
      float n[32];
      float rstd = 0.f;
      if (valid) {
        const float2 st = p.zstat[pr];
        rstd = st.x;
        load32_bf16(p.z + pr * kC + c0, n);
#pragma unroll
        for (int e = 0; e < 32; ++e) n[e] = fmaf(n[e], st.x, st.y);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) n[e] = 0.f;
      }
      float s1 = 0.f, s2 = 0.f;
      {
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float dn = dzh[e] * g_in[c0 + e];
          s1 += dn;
          s2 = fmaf(dn, n[e], s2);
          v[e] = dzh[e] * n[e];
        }
        acc_g += reduce_scatter32(v, lane);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = dzh[e];
        acc_b += reduce_scatter32(v, lane);
      }
      sm.sst[h][r] = make_float2(s1, s2);
      __syncthreads();
      {
        const float2 q0 = sm.sst[0][r], q1 = sm.sst[1][r], q2 = sm.sst[2][r], q3 = sm.sst[3][r];
        s1 = ((q0.x + q1.x) + (q2.x + q3.x)) * (1.f / kC);
        s2 = ((q0.y + q1.y) + (q2.y + q3.y)) * (1.f / kC);
      }
      if (valid) {
        float o[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = rstd * (dzh[e] * g_in[c0 + e] - s1 - n[e] * s2);
        uint4* dzp = reinterpret_cast<uint4*>(p.dz + pr * kC + c0);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          dzp[u] = make_uint4(pack_bf16x2(o[8 * u], o[8 * u + 1]), pack_bf16x2(o[8 * u + 2], o[8 * u + 3]),
                              pack_bf16x2(o[8 * u + 4], o[8 * u + 5]), pack_bf16x2(o[8 * u + 6], o[8 * u + 7]));
      }
    }
  }

  // per-CTA partial sums, added to
  if (ok && local > 0) {
    if (p.final_pass) {
      sm.red[lq][c0 + lane] = acc_g;
      sm.red[lq][kC + c0 + lane] = acc_b;
      __syncthreads();
      for (int k = tid; k < 2 * kC; k += NT)
        p.part_ln[(long long)blockIdx.x * 2 * kC + k] += ((sm.red[0][k] + sm.red[1][k]) + sm.red[2][k]) + sm.red[3][k];
    }
    float* pw = p.part_w + (long long)blockIdx.x * 2 * kC * kC + (long long)r * kC + c0;
#pragma unroll 1
    for (int mm = 0; mm < 2; ++mm) {
      uint32_t rr[32];
      tmem_ld32(trow + (2 + mm) * kC + c0, rr);
      tmem_ld_wait();
      const float u = mm == 0 ? u3 : u4;
#pragma unroll
      for (int e = 0; e < 32; ++e) pw[mm * kC * kC + e] += __uint_as_float(rr[e]) * u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Largest |value| of a bf16 tensor of n elements (n a multiple of 8, 16-byte aligned), merged into
// *out with an atomic maximum on the float's bits (non-negative floats order like their bits).
__global__ void __launch_bounds__(256) k_absmax_bf16(const __nv_bfloat16* __restrict__ v, long long n,
                                                      unsigned* out) {
  __shared__ unsigned red[8];
  uint32_t mx = 0;   // largest |bf16| as its bits (sign cleared)
  const uint4* q = reinterpret_cast<const uint4*>(v);
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n / 8; k += (long long)gridDim.x * blockDim.x) {
    const uint4 w = q[k];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = max(mx, max(ws[e] & 0x7fffu, (ws[e] >> 16) & 0x7fffu));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = max(mx, red[w]);
    atomicMax(out, mx << 16);   // the bf16 bits are the upper half of the float's
  }
}

}  // namespace

constexpr size_t kOutSmemBytes = sizeof(OutSmem) + 1024;
constexpr size_t kProjSmemBytes = sizeof(ProjSmem) + 1024;
static_assert(kOutSmemBytes <= 232448, "output backward shared memory");
static_assert(kProjSmemBytes <= 232448, "projection backward shared memory");

int bwd_grid(long long tiles, int num_sms) { return (int)(tiles < num_sms ? tiles : num_sms); }

cudaError_t launch_bwd_output_bf16(const BwdOutParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_bwd_output, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmemBytes);
  if (e != cudaSuccess) return e;
  k_bwd_output<<<grid, NT, kOutSmemBytes, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_project_bf16(const BwdProjParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_bwd_project, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kProjSmemBytes);
  if (e != cudaSuccess) return e;
  k_bwd_project<<<grid, NT, kProjSmemBytes, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_absmax_bf16(const __nv_bfloat16* v, long long n, unsigned* out, int num_sms, cudaStream_t s) {
  if (n % 8) return cudaErrorInvalidValue;
  long long blocks = (n / 8 + 255) / 256;
  const long long cap = 8LL * num_sms;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  k_absmax_bf16<<<(int)blocks, 256, 0, s>>>(v, n, out);
  return cudaGetLastError();
}

}  // namespace tmk
