// k_attention.cu -- triangle attention (starting and ending node) on the tensor cores, c_z = 128,
// H = 4 heads of c = 32.
//
// The BioIR page ("BioIR da Nvidia acelera previsão de proteínas em 2,9x com PyTorch puro") names
// triangle operations and pairwise attention among the Pairformer parts its kernels target; the
// arithmetic is the AlphaFold3 / Boltz triangle attention around the starting node:
//   zh = LN(z);  q, k, v, g = W_q zh, W_k zh, W_v zh, sigmoid(W_g zh);  b^h_jk = W_b^h zh_jk
//   o_ij^h = g_ij^h * sum_k softmax_k(q_ij^h . k_ik^h / sqrt(c) + b_jk^h) v_ik^h  over keys m_i m_k = 1
//   out_ij = W_o [o_ij^1 .. o_ij^H]
// and the ending node is the same on the transposed grid (z_ji in, out_ji written).
//
// Every intermediate (zh, q, k, v, g, the bias, the softmax weights P and the gated output o) is
// stored as fp16, whose 11 significant bits keep the path's error well inside the bf16 tolerance of
// the result (bf16 intermediates, 8 bits, cost several times more). zh and v (and with it o) are
// stored times powers of two that the host derives from bounds the weights fix, so that their
// largest possible values sit near 2^14 and small ones stay normal; q, k and the bias enter the
// logits, whose precision is absolute, and are stored as they are (the host refuses weights that
// could push them past 2^15).
//
// Three kernels.
//   k_ta_project: per tile of 128 pairs (512 threads, four per pair), LayerNorm statistics from the
//     pair's four channel quarters, zh into a 128 x 128 fp16 tile, one MMA each for q, k, v, g
//     (TMEM columns 0..511; weights as fp16 images scaled by a power of two each), b on the CUDA
//     cores. q, k and g are stored pair-major like z; v is stored per (row, head, channel) with the
//     key index innermost, so that it is the K-major operand of the P V product; b per (head, j) with
//     k innermost.
//   k_ta_attend: per (row i, block of 128 queries j), heads one after another, keys in blocks of 128:
//     S = Q K^T (tcgen05, TMEM; q stored times log2(e)/sqrt(c), the bias times log2(e), so the softmax
//     runs in base 2), + bias tile (-inf at masked keys), online softmax in registers (two threads per
//     query row, 64 keys each), P (fp16) into shared memory, O_blk = P V (tcgen05, with a row of ones
//     appended to v so that the product also gives the row sum of P, the softmax denominator) added
//     into the row's running output, the gate at the end of each head. Loads and products are pipelined one
//     block ahead: the next block's K and bias are fetched once this block's S and bias are in
//     registers, its S is issued together with this block's P V, and its v once P V is done.
//   k_ta_out: out = W_o o per pair (the ending node writes the transposed pair).
#include "pair_tile.cuh"

namespace tmk {
namespace {

using namespace pt;

constexpr int kHeads = 4, kHd = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQScale = 1.4426950408889634f * 0.17677669529663687f;   // log2(e) / sqrt(32)

struct alignas(1024) TaProjSmem {
  uint8_t zh[TILE], wq[TILE], wk[TILE], wv[TILE], wg[TILE];
  float ln[2 * kC];                    // gamma, beta
  float wb[kHeads * kC];               // W_b, float32
  float2 zst[4][BT];                   // per channel quarter and pair: (mean, M2) of z
  float bpart[4][kHeads][BT];          // per channel quarter: partial W_b zh
  uint64_t bar;
  uint32_t tmem_slot;
  int abort_flag;
};

__global__ void __launch_bounds__(NT, 1) k_ta_project(const TaProjectParams p) {
  extern __shared__ uint8_t smem_raw[];
  TaProjSmem& sm = *reinterpret_cast<TaProjSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lq = warp & 3, h = warp >> 2;   // TMEM lane quarter; channel quarter = head
  const int r = 32 * lq + lane;
  const int c0 = 32 * h;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  for (int k = tid; k < 2 * kC; k += NT) sm.ln[k] = p.ln[k];
  for (int k = tid; k < kHeads * kC; k += NT) sm.wb[k] = p.w_b[k];
  copy_tile(sm.wq, p.w_q);
  copy_tile(sm.wk, p.w_k);
  copy_tile(sm.wv, p.w_v);
  copy_tile(sm.wg, p.w_g);
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
  const uint32_t a_zh = smem_u32(sm.zh);

  uint32_t phase = 0;
  for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x) {
    const long long pr = t * BT + r;          // pair (i, j) of the (possibly transposed) grid
    const bool valid = pr < p.P;
    const int i = valid ? (int)(pr / p.N) : 0;
    const int j = valid ? (int)(pr - (long long)i * p.N) : 0;
    const long long zp = p.transpose ? (long long)j * p.N + i : pr;   // the z pair it reads

    // ---- LayerNorm of z: quarter statistics combined over the pair's four threads
    float f[32];
    if (valid) load32_bf16(p.z + zp * kC + c0, f);
    else
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = 0.f;
    {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) s += f[e];
      const float m = s * (1.f / 32);
      float m2 = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) m2 = fmaf(f[e] - m, f[e] - m, m2);
      sm.zst[h][r] = make_float2(m, m2);
    }
    __syncthreads();
    float mu, rs;
    {
      const float2 q0 = sm.zst[0][r], q1 = sm.zst[1][r], q2 = sm.zst[2][r], q3 = sm.zst[3][r];
      mu = ((q0.x + q1.x) + (q2.x + q3.x)) * 0.25f;
      const float d0 = q0.x - mu, d1 = q1.x - mu, d2 = q2.x - mu, d3 = q3.x - mu;
      const float m2 = ((q0.y + q1.y) + (q2.y + q3.y)) + 32.f * ((d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3));
      rs = rsqrtf(m2 * (1.f / kC) + 1e-5f);
    }
    float bp[kHeads] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      f[e] = valid ? sm.ln[c0 + e] * ((f[e] - mu) * rs) + sm.ln[kC + c0 + e] : 0.f;
#pragma unroll
      for (int hh = 0; hh < kHeads; ++hh) bp[hh] = fmaf(sm.wb[hh * kC + c0 + e], f[e], bp[hh]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) put8h(sm.zh, r, c0 + 8 * u, f + 8 * u);
#pragma unroll
    for (int hh = 0; hh < kHeads; ++hh) sm.bpart[h][hh][r] = bp[hh];
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma_tile(tmem, a_zh, false, smem_u32(sm.wq), false, ID_KK_H, false);
      mma_tile(tmem + kC, a_zh, false, smem_u32(sm.wk), false, ID_KK_H, false);
      mma_tile(tmem + 2 * kC, a_zh, false, smem_u32(sm.wv), false, ID_KK_H, false);
      mma_tile(tmem + 3 * kC, a_zh, false, smem_u32(sm.wg), false, ID_KK_H, false);
      mma_commit(&sm.bar);
    }
    // b of head h for this pair: the four quarters' partial sums
    if (valid) {
      // the bias of query i and key j; a masked key j gets -inf, which removes it from every softmax
      const float bsum = ((sm.bpart[0][h][r] + sm.bpart[1][h][r]) + sm.bpart[2][h][r]) + sm.bpart[3][h][r];
      const bool kmasked = p.mask && p.mask[j] == 0.f;
      p.b[((long long)h * p.N + i) * p.ldb + j] = __float2half_rn(kmasked ? -INFINITY : bsum * p.bscale);
    }
    if (!cta_wait(&sm.bar, phase, p.w, &sm.abort_flag, 1)) break;
    phase ^= 1u;
    tc_fence_after();

    // ---- q, k, g pair-major (this head's 32 channels); v per (row, head, channel), key innermost
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      uint32_t rr[32];
      tmem_ld32(trow + m * kC + c0, rr);
      tmem_ld_wait();
      if (!valid) continue;
      float o[32];
      // undoes the weight image's power-of-two scale; q's also carries log2(e)/sqrt(c), so that q . k is
      // the logit in the base-2 exponent of the softmax
      const float sc = p.wscale[m];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = __uint_as_float(rr[e]) * sc;
        o[e] = m == 3 ? sigmoid_mufu(x) : x;
      }
      if (m == 2) {
        __half* vp = p.vt + ((long long)i * kC + c0) * p.ldv + j;
#pragma unroll
        for (int e = 0; e < 32; ++e) vp[(long long)e * p.ldv] = __float2half_rn(o[e]);
      } else {
        __half* dst = (m == 0 ? p.q : m == 1 ? p.k : p.g) + pr * kC + c0;
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int u = 0; u < 4; ++u) d4[u] = pack8h(o + 8 * u);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

namespace {

constexpr uint32_t kQBytes = 64 * 128 * 2;      // Q box: 64 channels (a head pair) x 128 queries
constexpr uint32_t kKBytes = 64 * 128 * 2;      // K box: 64 channels x 128 keys
constexpr uint32_t kVBytes = 64 * 32 * 2;       // one v box: 64 keys x 32 channels of one head
constexpr uint32_t kVSlot = 64 * 48 * 2;        // its slot: 32 rows of v, a row of ones, 15 rows of zeros
constexpr int kPvN = 48;                        // N of the P V product: 32 channels, the row sum, padding
constexpr uint32_t kBBytes = 64 * 128 * 2;      // one bias box: 64 keys x 128 queries

static_assert(kBoxTaQK.bytes() == kQBytes && kBoxTaQK.bytes() == kKBytes, "Q/K box fills its slot");
static_assert(kBoxTaV.bytes() == kVBytes, "v box fills its slot");
static_assert(kBoxTaBias.bytes() == kBBytes, "bias box fills its slot");

struct alignas(1024) TaAttSmem {
  uint8_t q[kQBytes];
  uint8_t k[kKBytes];
  uint8_t b[2][kBBytes];                        // keys 0..63 and 64..127 of the block
  uint8_t p[TILE];                              // P: 128 queries x 128 keys, fp16, K-major
  uint8_t v[2][kVSlot];                         // keys 0..63 and 64..127, rows = channels (+ ones row)
  float xmax[2][BT];                            // per key half and query: block maximum
  uint64_t kb_bar, v_bar, s_bar, pv_bar;
  uint32_t tmem_slot;
  int abort_flag;
};

constexpr int kAttThreads = 256;   // two threads per query row, 64 keys of each block each

__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

__global__ void __launch_bounds__(kAttThreads, 2) k_ta_attend(const __grid_constant__ CUtensorMap qmap,
                                                              const __grid_constant__ CUtensorMap kmap,
                                                              const __grid_constant__ CUtensorMap vmap,
                                                              const __grid_constant__ CUtensorMap bmap,
                                                              const TaAttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  TaAttSmem& sm = *reinterpret_cast<TaAttSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = 32 * (warp & 3) + lane;      // query row of the block (TMEM lane)
  const int kh = warp >> 2;                    // key half of every block; output channels 16 kh ..
  const int i = (int)(blockIdx.x / p.jblocks);
  const int jb = (int)(blockIdx.x - (long long)i * p.jblocks);
  const int j = jb * BT + row;
  const bool jvalid = j < p.N;
  __half* orow = p.o + ((long long)i * p.N + j) * kC;
  if (p.mask && p.mask[i] == 0.f) {
    // no valid key in this row: o = 0
    if (jvalid) {
      uint4* d = reinterpret_cast<uint4*>(orow) + 8 * kh;
#pragma unroll
      for (int u = 0; u < 8; ++u) d[u] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  const int kblocks = (p.N + BT - 1) / BT;
  const int total = kHeads * kblocks;          // iterations: heads in order, key blocks within a head
  // loads of iteration t: K and bias (and Q at the start of a head pair) on kb_bar, v on v_bar
  auto load_kb = [&](int t) {
    const int h = t / kblocks, kb = t - h * kblocks;
    const bool with_q = kb == 0 && (h & 1) == 0;
    mbar_expect_tx(&sm.kb_bar, kKBytes + 2 * kBBytes + (with_q ? kQBytes : 0u));
    if (with_q) tma_load_3d(sm.q, &qmap, &sm.kb_bar, 64 * (h >> 1), jb * BT, i);
    tma_load_3d(sm.k, &kmap, &sm.kb_bar, 64 * (h >> 1), kb * BT, i);
    tma_load_3d(sm.b[0], &bmap, &sm.kb_bar, kb * BT, jb * BT, h);
    tma_load_3d(sm.b[1], &bmap, &sm.kb_bar, kb * BT + 64, jb * BT, h);
  };
  auto load_v = [&](int t) {
    const int h = t / kblocks, kb = t - h * kblocks;
    mbar_expect_tx(&sm.v_bar, 2 * kVBytes);
    tma_load_3d(sm.v[0], &vmap, &sm.v_bar, kb * BT, kHd * h, i);
    tma_load_3d(sm.v[1], &vmap, &sm.v_bar, kb * BT + 64, kHd * h, i);
  };
  constexpr uint32_t ID_S = make_idesc(128, 128, FMT_F16, false, false);
  constexpr uint32_t ID_O = make_idesc(128, kPvN, FMT_F16, false, false);
  auto issue_s = [&](uint32_t tmem, int t) {     // S = Q_h K_h^T (q is stored pre-scaled by log2(e)/sqrt(c))
    const int hh = (t / kblocks) & 1;
    const uint32_t q0 = smem_u32(sm.q) + 64 * hh, k0 = smem_u32(sm.k) + 64 * hh;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
      mma_f16(tmem, make_sdesc_sw128(q0 + 32 * ks, 16, 1024), make_sdesc_sw128(k0 + 32 * ks, 16, 1024), ID_S,
              ks ? 1u : 0u);
    mma_commit(&sm.s_bar);
  };

  if (tid == 0) {
    mbar_init(&sm.kb_bar, 1);
    mbar_init(&sm.v_bar, 1);
    mbar_init(&sm.s_bar, 1);
    mbar_init(&sm.pv_bar, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&bmap);
    load_kb(0);
    load_v(0);
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_slot, 256);
    tmem_relinquish();
  }
  // rows 32..47 of both v slots, which no copy overwrites: a row of ones (the P V product's column 32
  // is then the row sum of the bf16 P, the softmax denominator) and zeros
  for (int x = tid; x < 2 * (kVSlot - kVBytes) / 4; x += kAttThreads) {
    const int half = x / ((kVSlot - kVBytes) / 4), w4 = x % ((kVSlot - kVBytes) / 4);
    reinterpret_cast<uint32_t*>(sm.v[half] + kVBytes)[w4] = w4 < 32 ? 0x3C003C00u : 0u;   // fp16 1.0 pairs
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  uint32_t kph = 0, vph = 0, sph = 0, pph = 0;   // phases (kb/v: thread 0 only)
  bool ok = true;
  if (tid == 0) {
    if (wait_bounded(&sm.kb_bar, kph, p.w, &sm.abort_flag, 1)) {
      tc_fence_after();
      issue_s(tmem, 0);
    }
    kph ^= 1u;
  }

  float m_run = -INFINITY, l_run = 0.f;
  float acc[16];
  for (int t = 0; t < total; ++t) {
    const int h = t / kblocks, kb = t - h * kblocks;
    if (kb == 0) {
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    }
    if (!cta_wait(&sm.s_bar, sph, p.w, &sm.abort_flag, 2)) { ok = false; break; }
    sph ^= 1u;
    tc_fence_after();

    // ---- this thread's 64 logits (log2 domain): S + b, b stored times log2(e) and -inf at masked keys;
    // keys past the grid (last block only) -> -inf
    // every thread observes the completion of this block's bias copy before reading it (load t is the
    // t-th completion of kb_bar; load t + 1 is issued only after all threads are past this point)
    if (!wait_bounded(&sm.kb_bar, (uint32_t)(t & 1), p.w, &sm.abort_flag, 8)) ok = false;
    float sv[64];
    {
      uint32_t r0[32], r1[32];
      tmem_ld32(trow + 64 * kh, r0);
      tmem_ld32(trow + 64 * kh + 32, r1);
      tmem_ld_wait();
      const uint8_t* brow = sm.b[kh];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float bv[8];
        f16x8_to_float(*reinterpret_cast<const uint4*>(brow + sw128_offset((uint32_t)row, (uint32_t)u)), bv);
#pragma unroll
        for (int e = 0; e < 8; ++e) sv[8 * u + e] = __uint_as_float(u < 4 ? r0[8 * u + e] : r1[8 * (u - 4) + e]) + bv[e];
      }
    }
    if (kb == kblocks - 1) {
      const int kbase = kb * BT + 64 * kh;
#pragma unroll
      for (int e = 0; e < 64; ++e)
        if (kbase + e >= p.N) sv[e] = -INFINITY;
    }
    float bmax = sv[0];
#pragma unroll
    for (int e = 1; e < 64; ++e) bmax = fmaxf(bmax, sv[e]);
    sm.xmax[kh][row] = bmax;
    tc_fence_before();
    __syncthreads();
    // S, K and the bias of this block have been read: the next block's K and bias can come in
    if (tid == 0 && t + 1 < total) load_kb(t + 1);
    const float m_new = fmaxf(m_run, fmaxf(sm.xmax[0][row], sm.xmax[1][row]));
    const float mref = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2_approx(m_run - mref);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) pv[e] = ex2_approx(sv[8 * u + e] - mref);
      put8h(sm.p, row, 64 * kh + 8 * u, pv);
    }
    m_run = m_new;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      // P V of this block, then S of the next one (different TMEM columns, different operands)
      if (wait_bounded(&sm.v_bar, vph, p.w, &sm.abort_flag, 3)) {
        const uint32_t p0 = smem_u32(sm.p), v0 = smem_u32(sm.v[0]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_f16(tmem + BT, make_sdesc_sw128(p0 + (ks >> 2) * SLAB + (ks & 3) * 32, 16, 1024),
                  make_sdesc_sw128(v0 + (ks >> 2) * kVSlot + (ks & 3) * 32, 16, 1024), ID_O, ks ? 1u : 0u);
        mma_commit(&sm.pv_bar);
      }
      vph ^= 1u;
      if (t + 1 < total) {
        if (wait_bounded(&sm.kb_bar, kph, p.w, &sm.abort_flag, 4)) {
          tc_fence_after();
          issue_s(tmem, t + 1);
        }
        kph ^= 1u;
      }
    }
    if (!cta_wait(&sm.pv_bar, pph, p.w, &sm.abort_flag, 5)) { ok = false; break; }
    pph ^= 1u;
    tc_fence_after();
    // P V has read v: the next block's v can come in
    if (tid == 0 && t + 1 < total) load_v(t + 1);
    {
      uint32_t ro[16];
      tmem_ld16(trow + BT + 16 * kh, ro);
      const uint32_t rl = tmem_ld1(trow + BT + kHd);     // the row sum of this block's P
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = fmaf(acc[e], alpha, __uint_as_float(ro[e]));
      l_run = fmaf(l_run, alpha, __uint_as_float(rl));
    }
    if (kb == kblocks - 1) {
      // ---- o = g * acc / l for 16 channels of head h (l: the running sum of the bf16 P over all keys)
      const float l_tot = l_run;
      if (jvalid) {
        const int cb = kHd * h + 16 * kh;
        float gv[16];
        {
          const uint4* gq = reinterpret_cast<const uint4*>(p.g + ((long long)i * p.N + j) * kC + cb);
          const uint4 g0 = gq[0], g1 = gq[1];
          f16x8_to_float(g0, gv);
          f16x8_to_float(g1, gv + 8);
        }
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        float o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = gv[e] * acc[e] * inv;
        uint4* d4 = reinterpret_cast<uint4*>(orow + cb);
#pragma unroll
        for (int u = 0; u < 2; ++u) d4[u] = pack8h(o + 8 * u);
      }
    }
  }
  if (!ok && tid == 0) {
    // a wait ran out: let copies still in flight land before the shared memory is released
    wait_bounded(&sm.kb_bar, kph, p.w, &sm.abort_flag, 6);
    wait_bounded(&sm.v_bar, vph, p.w, &sm.abort_flag, 7);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// out = W_o o per pair (512 threads, tiles of 128 pairs; o and the W_o image fp16); for the ending
// node the pair (i, j) of the transposed grid is written at (j, i).
struct alignas(1024) TaOutSmem {
  uint8_t o[TILE], wo[TILE];
  uint64_t bar;
  uint32_t tmem_slot;
  int abort_flag;
};

__global__ void __launch_bounds__(NT, 1) k_ta_out(const TaOutParams p) {
  extern __shared__ uint8_t smem_raw[];
  TaOutSmem& sm = *reinterpret_cast<TaOutSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lq = warp & 3, h = warp >> 2;
  const int r = 32 * lq + lane;
  const int c0 = 32 * h;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  copy_tile(sm.wo, p.w_o);
  if (warp == 0) {
    tmem_alloc(&sm.tmem_slot, 128);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)(32 * lq) << 16);
  uint32_t phase = 0;
  for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x) {
    const long long pr = t * BT + r;
    const bool valid = pr < p.P;
    const int i = valid ? (int)(pr / p.N) : 0;
    const int j = valid ? (int)(pr - (long long)i * p.N) : 0;
    float f[32];
    if (valid) load32_f16(p.o + pr * kC + c0, f);
    else
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) put8h(sm.o, r, c0 + 8 * u, f + 8 * u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma_tile(tmem, smem_u32(sm.o), false, smem_u32(sm.wo), false, ID_KK_H, false);
      mma_commit(&sm.bar);
    }
    if (!cta_wait(&sm.bar, phase, p.w, &sm.abort_flag, 1)) break;
    phase ^= 1u;
    tc_fence_after();
    uint32_t rr[32];
    tmem_ld32(trow + c0, rr);
    tmem_ld_wait();
    if (valid) {
      const long long op = p.transpose ? (long long)j * p.N + i : pr;
      uint4* d4 = reinterpret_cast<uint4*>(p.out + op * kC + c0);
      const float sc = p.oscale;    // undoes the power-of-two scale of the W_o image
#pragma unroll
      for (int u = 0; u < 4; ++u)
        d4[u] = make_uint4(pack_bf16x2(__uint_as_float(rr[8 * u]) * sc, __uint_as_float(rr[8 * u + 1]) * sc),
                           pack_bf16x2(__uint_as_float(rr[8 * u + 2]) * sc, __uint_as_float(rr[8 * u + 3]) * sc),
                           pack_bf16x2(__uint_as_float(rr[8 * u + 4]) * sc, __uint_as_float(rr[8 * u + 5]) * sc),
                           pack_bf16x2(__uint_as_float(rr[8 * u + 6]) * sc, __uint_as_float(rr[8 * u + 7]) * sc));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

constexpr size_t kTaProjSmem = sizeof(TaProjSmem) + 1024;
constexpr size_t kTaAttSmem = sizeof(TaAttSmem) + 1024;
constexpr size_t kTaOutSmem = sizeof(TaOutSmem) + 1024;
static_assert(kTaProjSmem <= 232448, "attention projection shared memory");
static_assert(2 * kTaAttSmem <= 233472, "two attention CTAs per SM");
static_assert(kTaOutSmem <= 232448, "attention output shared memory");

cudaError_t launch_ta_project(const TaProjectParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_ta_project, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTaProjSmem);
  if (e != cudaSuccess) return e;
  k_ta_project<<<grid, NT, kTaProjSmem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ta_attend(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const CUtensorMap& bmap, const TaAttendParams& p, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_ta_attend, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTaAttSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.jblocks;
  k_ta_attend<<<(unsigned)grid, kAttThreads, kTaAttSmem, s>>>(qmap, kmap, vmap, bmap, p);
  return cudaGetLastError();
}

cudaError_t launch_ta_out(const TaOutParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_ta_out, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTaOutSmem);
  if (e != cudaSuccess) return e;
  k_ta_out<<<grid, NT, kTaOutSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tmk
