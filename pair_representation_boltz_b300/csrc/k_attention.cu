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
//   k_ta_attend: per (row i, two tiles of 128 queries j), heads one after another, keys in blocks of
//     64, warp-specialised: a TMA warp, one MMA warp per query tile and one softmax thread per query
//     row. S = Q K^T (tcgen05, TMEM, three buffers per tile so that S runs up to three blocks ahead; q
//     stored times log2(e)/sqrt(c), the bias times log2(e), so the softmax runs in base 2); the softmax
//     thread reads its S row of the block with two TMEM loads under one wait, adds the bias row (-inf
//     at masked keys) and forms P = 2^(x - reference) against a lazy running reference while it takes
//     the block maximum (P again, from the logits in registers, only when the maximum moved by more
//     than 8), and stores P as fp16 over the S it has read; O += P v (A = P from TMEM, v with a row of
//     ones appended so that the product also gives the row sum of P, the softmax denominator)
//     accumulates across a head's blocks in TMEM, and the gate is applied at the end of each head.
//   k_ta_out: out = W_o o per pair (the ending node writes the transposed pair).
#include "pair_tile.cuh"

namespace tmk {
namespace {

using namespace pt;

constexpr int kHeads = 4, kHd = 32;

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
    if (!p.transpose) {
      // L2 prefetch of the CTA's next tile of z: its pairs' rows are one contiguous run (one request)
      const long long n0 = (t + gridDim.x) * BT;
      if (tid == 0 && n0 < p.P) {
        const long long n1 = n0 + BT < p.P ? n0 + BT : p.P;
        prefetch_l2_bulk(p.z + n0 * kC, (uint32_t)((n1 - n0) * kC * 2));
      }
    } else {
      // transposed, the rows of the next tile lie N rows apart: one request per pair, by its first thread
      const long long pn = pr + (long long)gridDim.x * BT;
      if (h == 0 && pn < p.P) {
        const int in = (int)(pn / p.N), jn = (int)(pn - (long long)in * p.N);
        prefetch_l2_bulk(p.z + ((long long)jn * p.N + in) * kC, kC * 2);
      }
    }

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

constexpr int kKB = 64;                         // keys per block
constexpr uint32_t kQBytes = 64 * 128 * 2;      // Q box: 64 channels (a head pair) x 128 queries
constexpr uint32_t kKBytes = 64 * kKB * 2;      // K box: 64 channels x 64 keys
constexpr uint32_t kVBytes = kKB * 32 * 2;      // v box: 64 keys x 32 channels of one head
constexpr uint32_t kVSlot = kKB * 48 * 2;       // its slot: 32 rows of v, a row of ones, 15 rows of zeros
constexpr int kPvN = 48;                        // N of the P V product: 32 channels, the row sum, padding
constexpr uint32_t kBBytes = kKB * 128 * 2;     // one bias box: 64 keys x 128 queries

static_assert(kBoxTaQK.bytes() == kQBytes, "Q box fills its slot");
static_assert(kBoxTaK.bytes() == kKBytes, "K box fills its slot");
static_assert(kBoxTaV.bytes() == kVBytes, "v box fills its slot");
static_assert(kBoxTaBias.bytes() == kBBytes, "bias box fills its slot");

constexpr int kGroups = 2;            // query tiles per CTA, one softmax group each
constexpr int kStages = 4;            // K, v and bias stages in flight
constexpr int kSBuf = 3;              // S (and P) buffers per group in TMEM
constexpr int kAttThreads = 32 + 32 * kGroups + 32 * 4 * kGroups;   // TMA warp, an MMA warp and four softmax warps per group
constexpr uint32_t kStageBytes = kKBytes + kGroups * kBBytes + kVBytes;   // what one stage receives

struct alignas(1024) TaAttSmem {
  uint8_t q[kGroups][kQBytes];                  // per group: 64 channels (a head pair) x 128 queries
  uint8_t k[kStages][kKBytes];                  // 64 channels x 64 keys
  uint8_t b[kStages][kGroups][kBBytes];         // bias: per group, the block's 64 keys x 128 queries
  uint8_t v[kStages][kVSlot];                   // the block's 64 keys, rows = channels (+ ones row)
  uint64_t q_full, q_free, go1;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kGroups][kSBuf], p_full[kGroups][kSBuf], pv_done[kGroups][2], pv_last[kGroups], fin[kGroups];
  uint32_t tmem_slot;
  int abort_flag;
};

// TMEM columns of group g (base 256 g): the three block buffers at 0, 64 and 128, each S (64 keys,
// float32) and then, over its first 32 columns, P (64 keys as packed fp16 pairs) once S has been read;
// the running output P V (32 channels, the row sum, padding) at 192.
constexpr uint32_t kTmS = 0, kTmPV = 192, kTmGroup = 256;
static_assert(kSBuf * kKB <= (int)kTmPV, "S buffers below the running output");

// Non-blocking probe of a barrier phase (acquire when it reports completion): the result can be consumed
// later, so the probe's latency overlaps other work.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Triangle attention of one CTA: row i of the grid, query tiles 2 jp and 2 jp + 1 (one per softmax
// group), heads in turn, keys in blocks of 64. Roles:
//   warp 0        TMA: per block, K (the head pair's 64 channels), the bias tiles of both groups and
//                 v (with a row of ones beside it) into one of four stages; Q of both groups per head pair.
//   warps 1, 2    tcgen05.mma for group g = warp - 1: S_g = Q_g K^T into one of three TMEM buffers
//                 (M = 128 queries, N = 64 keys, K = 32), up to three blocks ahead of the softmax, and,
//                 once the group has stored P of a block over its S, O_g += P_g v (A = P from TMEM, B = v
//                 from shared memory, N = 48: 32 channels, the row sum from the ones row, padding). The
//                 product of block t is issued before S of block t + 3 into the same buffer: the tensor
//                 core runs one thread's MMAs in order, so S of a block complete means every product up
//                 to three blocks back is complete. Operand descriptors are the tile's plus an offset, and
//                 the block, stage and buffer indices advance as counters (no division per block).
//   warps 3..10   softmax, thread = query row, group g = the four warps of one query tile: S row +
//                 bias row -> logits (base 2), and P = 2^(x - m) against the row's running reference
//                 m, formed while the block maximum is taken. The reference is lazy: it moves only when
//                 the maximum exceeds it by more than 8 (always at a head's first block; P is then formed
//                 again from the logits still in registers), so P <= 2^8 stays inside fp16 and most
//                 blocks leave the running output as it is. P goes into TMEM as fp16 over the first half
//                 of the block's S columns. The running output O (and its row sum) accumulates in TMEM
//                 across a head's blocks; when the reference moves, the thread rescales its row of O once
//                 the block before has been added, before this block's P is released. The second group
//                 starts one block behind the first. Each block probes the next block's S and bias
//                 barriers without blocking once its logits are in registers; when both had completed,
//                 the next block skips its two waits (about 1 % of the kernel's time).
__global__ void __launch_bounds__(kAttThreads, 1) k_ta_attend(const __grid_constant__ CUtensorMap qmap,
                                                              const __grid_constant__ CUtensorMap kmap,
                                                              const __grid_constant__ CUtensorMap vmap,
                                                              const __grid_constant__ CUtensorMap bmap,
                                                              const TaAttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  TaAttSmem& sm = *reinterpret_cast<TaAttSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = (int)(blockIdx.x / p.jpairs);
  const int jp = (int)(blockIdx.x - (long long)i * p.jpairs);
  if (p.mask && p.mask[i] == 0.f) {
    // no valid key in this row: o = 0 for every query of both tiles
    for (int u = tid; u < kGroups * BT * (kC / 8); u += kAttThreads) {
      const int jq = jp * kGroups * BT + u / (kC / 8);
      if (jq < p.N) reinterpret_cast<uint4*>(p.o + ((long long)i * p.N + jq) * kC)[u % (kC / 8)] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  const int KB = (p.N + kKB - 1) / kKB;
  const int T = 4 * KB;                          // iterations: heads in order, key blocks within a head

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, kGroups);              // each group's MMA warp
    mbar_init(&sm.go1, 4);                       // group 0 has finished its first block
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&sm.kv_full[st], 1);
      mbar_init(&sm.kv_empty[st], kGroups + 4 * kGroups);   // each MMA warp's commit + every softmax warp (bias read)
    }
    for (int g = 0; g < kGroups; ++g) {
      for (int b = 0; b < kSBuf; ++b) {
        mbar_init(&sm.s_full[g][b], 1);
        mbar_init(&sm.p_full[g][b], 4);
      }
      mbar_init(&sm.pv_done[g][0], 1);
      mbar_init(&sm.pv_done[g][1], 1);
      mbar_init(&sm.pv_last[g], 1);
      mbar_init(&sm.fin[g], 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_slot, 512);
    tmem_relinquish();
  }
  // rows 32..47 of every v slot, which no copy overwrites: a row of ones (the P V product's column 32
  // is then the row sum of the fp16 P, the softmax denominator) and zeros
  for (int x = tid; x < kStages * (int)((kVSlot - kVBytes) / 4); x += kAttThreads) {
    const int slot = x / (int)((kVSlot - kVBytes) / 4), w4 = x % (int)((kVSlot - kVBytes) / 4);
    reinterpret_cast<uint32_t*>(sm.v[slot] + kVBytes)[w4] = w4 < 32 ? 0x3C003C00u : 0u;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      tma_prefetch_desc(&bmap);
      for (int t = 0; t < T; ++t) {
        const int h = t / KB, kb = t - h * KB, st = t % kStages, use = t / kStages;
        if (kb == 0 && (h & 1) == 0) {
          // Q of the head pair; the second pair's replaces the first once every S of heads 0, 1 is done
          if (h == 2 && !wait_bounded(&sm.q_free, 0, p.w, abort_flag, 11)) break;
          mbar_expect_tx(&sm.q_full, kGroups * kQBytes);
          for (int g = 0; g < kGroups; ++g)
            tma_load_3d(sm.q[g], &qmap, &sm.q_full, 64 * (h >> 1), (jp * kGroups + g) * BT, i);
        }
        if (use >= 1 && !wait_bounded(&sm.kv_empty[st], (uint32_t)(use - 1) & 1u, p.w, abort_flag, 12)) break;
        mbar_expect_tx(&sm.kv_full[st], kStageBytes);
        tma_load_3d(sm.k[st], &kmap, &sm.kv_full[st], 64 * (h >> 1), kb * kKB, i);
        for (int g = 0; g < kGroups; ++g)
          tma_load_3d(sm.b[st][g], &bmap, &sm.kv_full[st], kb * kKB, (jp * kGroups + g) * BT, h);
        tma_load_3d(sm.v[st], &vmap, &sm.kv_full[st], kb * kKB, kHd * h, i);
      }
    }
  } else if (warp <= kGroups) {
    // ------------------------------------------------------------ MMA issuer of group g = warp - 1
    if (lane == 0) {
      const int g = warp - 1;
      constexpr uint32_t ID_S = make_idesc(128, kKB, FMT_F16, false, false);
      constexpr uint32_t ID_O = make_idesc(128, kPvN, FMT_F16, false, false);
      const uint32_t tg = tmem + (uint32_t)g * kTmGroup;
      // descriptors of the operand tiles at offset 0; an operand's descriptor is its tile's plus the
      // byte offset / 16 (the start-address field, shared memory below 256 KB)
      const uint64_t dq = make_sdesc_sw128(smem_u32(sm.q[g]), 16, 1024);
      const uint64_t dk = make_sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t dv = make_sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
      // block cursors: block t, its head h, key block kb, stage st with its use parity, S buffer b with its
      // use parity
      struct Cur {
        int t, h, kb, st, b;
        uint32_t sph, bph;
      };
      auto next = [&](Cur& c) {
        ++c.t;
        if (++c.kb == KB) { c.kb = 0; ++c.h; }
        if (++c.st == kStages) { c.st = 0; c.sph ^= 1u; }
        if (++c.b == kSBuf) { c.b = 0; c.bph ^= 1u; }
      };
      // S_g of the cursor's block into its buffer (q is stored pre-scaled by log2(e)/sqrt(c))
      auto issue_s = [&](const Cur& c) -> bool {
        if (c.kb == 0 && (c.h & 1) == 0 && !wait_bounded(&sm.q_full, (uint32_t)(c.h >> 1) & 1u, p.w, abort_flag, 20)) return false;
        if (!wait_bounded(&sm.kv_full[c.st], c.sph, p.w, abort_flag, 21)) return false;
        // the second group starts one block behind the first, so that each group's softmax overlaps
        // the other's wait for its products
        if (g == 1 && c.t == 0 && !wait_bounded(&sm.go1, 0u, p.w, abort_flag, 25)) return false;
        tc_fence_after();
        const uint32_t hoff = (uint32_t)(64 * (c.h & 1)) >> 4;
        const uint64_t aq = dq + hoff, bk = dk + ((uint32_t)c.st * (kKBytes >> 4) + hoff);
        const uint32_t dst = tg + kTmS + (uint32_t)(kKB * c.b);
        mma_f16(dst, aq, bk, ID_S, 0u);
        mma_f16(dst, aq + 2, bk + 2, ID_S, 1u);
        mma_commit(&sm.s_full[g][c.b]);
        if (c.t == 2 * KB - 1) mma_commit(&sm.q_free);   // every S of heads 0, 1 of this group issued
        return true;
      };
      // O_g (+)= P_g v of the cursor's block, once the group has stored P (and so has read S) of that
      // block. The tensor core runs a thread's MMAs in issue order, so S of the block three later, issued
      // next into the same buffer, overwrites P only after this product has read it.
      auto issue_pv = [&](const Cur& c) -> bool {
        if (!wait_bounded(&sm.p_full[g][c.b], c.bph, p.w, abort_flag, 23)) return false;
        tc_fence_after();
        const uint64_t bv = dv + (uint32_t)c.st * (kVSlot >> 4);
        const uint32_t pa = tg + kTmS + (uint32_t)(kKB * c.b);
        const uint32_t acc0 = c.kb != 0 ? 1u : 0u;    // a head's first block starts its running output
#pragma unroll
        for (int ks = 0; ks < kKB / 16; ++ks)
          mma_f16_ts(tg + kTmPV, pa + (uint32_t)(8 * ks), bv + (uint32_t)(2 * ks), ID_O, ks ? 1u : acc0);
        mma_commit(&sm.kv_empty[c.st]);    // this group's reads of K and v of the stage are done
        mma_commit(&sm.pv_done[g][c.t & 1]);
        return true;
      };
      Cur cs{0, 0, 0, 0, 0, 0u, 0u}, cp = cs;
      bool ok = true;
      for (int u = 0; u < kSBuf && ok; ++u, next(cs)) ok = issue_s(cs);
      for (; cp.t < T && ok; next(cp)) {
        ok = issue_pv(cp);
        if (ok && cs.t < T) {
          ok = issue_s(cs);
          next(cs);
        }
      }
      if (ok) mma_commit(&sm.pv_last[g]);   // every product of the group issued
      mma_commit(&sm.fin[g]);
      wait_bounded(&sm.fin[g], 0, p.w, abort_flag, 24);
    }
  } else {
    // ------------------------------------------------------------ softmax, thread = query row
    const int g = (warp - 1 - kGroups) >> 2;   // the group's query tile: 2 jp + g
    const int lq = warp & 3;                   // TMEM lane quarter
    const int row = 32 * lq + lane;
    const int j = (jp * kGroups + g) * BT + row;
    const bool jvalid = j < p.N;
    const uint32_t trow = tmem + ((uint32_t)(32 * lq) << 16) + (uint32_t)g * kTmGroup;
    float m_run = -INFINITY;
    // o = g * O / l for head hf, from the running output in TMEM (l: its column of the row sums of the fp16 P)
    auto finalize = [&](int hf) {
      uint32_t ro[32];
      tmem_ld32(trow + kTmPV, ro);
      const uint32_t rl = tmem_ld1(trow + kTmPV + kHd);
      tmem_ld_wait();
      if (!jvalid) return;
      const __half* gp = p.g + ((long long)i * p.N + j) * kC + kHd * hf;
      float gv[kHd];
#pragma unroll
      for (int u = 0; u < 4; ++u) f16x8_to_float(reinterpret_cast<const uint4*>(gp)[u], gv + 8 * u);
      const float l = __uint_as_float(rl);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float o[kHd];
#pragma unroll
      for (int e = 0; e < kHd; ++e) o[e] = gv[e] * __uint_as_float(ro[e]) * inv;
      uint4* d4 = reinterpret_cast<uint4*>(p.o + ((long long)i * p.N + j) * kC + kHd * hf);
#pragma unroll
      for (int u = 0; u < 4; ++u) d4[u] = pack8h(o + 8 * u);
    };
    // The block's S row (64 keys, two TMEM loads under one wait) into registers, as logits x = S + bias
    // (base 2; -inf past the grid's last key), and P = 2^(x - ref) packed as fp16 pairs into pk; returns
    // the logits' maximum.
    // byte offsets of the 16-byte units of this thread's bias row (128-byte swizzle)
    uint32_t boff[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) boff[u] = sw128_offset((uint32_t)row, (uint32_t)u);
    auto logits = [&](int st, int b, int nvalid, float ref, uint32_t (&r)[2][32], uint32_t (&pk)[2][16]) -> float {
      const float2 nref = make_float2(-ref, -ref);
      float mx = -INFINITY;
      tmem_ld32(trow + kTmS + kKB * b, r[0]);
      tmem_ld32(trow + kTmS + kKB * b + 32, r[1]);
      tmem_ld_wait();
      const uint8_t* brow = sm.b[st][g];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float bv[8];
          f16x8_to_float(*reinterpret_cast<const uint4*>(brow + boff[4 * cc + u]), bv);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 v = __fadd2_rn(make_float2(__uint_as_float(r[cc][8 * u + e]), __uint_as_float(r[cc][8 * u + e + 1])),
                                        make_float2(bv[e], bv[e + 1]));
            r[cc][8 * u + e] = __float_as_uint(v.x);
            r[cc][8 * u + e + 1] = __float_as_uint(v.y);
          }
        }
        if (nvalid < kKB) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * cc + e >= nvalid) r[cc][e] = __float_as_uint(-INFINITY);
        }
        float m3[11];
#pragma unroll
        for (int e = 0; e < 10; ++e)
          m3[e] = max3f(__uint_as_float(r[cc][3 * e]), __uint_as_float(r[cc][3 * e + 1]), __uint_as_float(r[cc][3 * e + 2]));
        m3[10] = max3f(__uint_as_float(r[cc][30]), __uint_as_float(r[cc][31]), mx);
        mx = max3f(max3f(m3[0], m3[1], m3[2]), max3f(m3[3], m3[4], m3[5]), max3f(max3f(m3[6], m3[7], m3[8]), m3[9], m3[10]));
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 d = __fadd2_rn(make_float2(__uint_as_float(r[cc][2 * e]), __uint_as_float(r[cc][2 * e + 1])), nref);
          pk[cc][e] = pack_f16x2(ex2_approx(d.x), ex2_approx(d.y));
        }
      }
      return mx;
    };
    bool ok = true;
    int h = 0, kb = 0, st = 0, b = 0;
    uint32_t sph = 0, bph = 0;
    bool probed = false;     // this block's S and bias barriers, probed during the block before
    for (int t = 0; t < T; ++t) {
      if (!__all_sync(0xffffffffu, probed)) {
        // S of this block is complete, and with it the P V product three blocks back
        if (!warp_wait_bounded(&sm.s_full[g][b], bph, p.w, abort_flag, 30)) { ok = false; break; }
        // every thread observes the completion of the stage's copies (the bias) before reading them
        if (!warp_wait_bounded(&sm.kv_full[st], sph, p.w, abort_flag, 31)) { ok = false; break; }
      }
      tc_fence_after();
      // ---- at a head's first block, the running output holds the head before's, complete once the
      // product of the block before is (the products up to three blocks back are)
      if (t >= 1 && kb == 0) {
        if (!warp_wait_bounded(&sm.pv_done[g][(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, p.w, abort_flag, 32)) { ok = false; break; }
        tc_fence_after();
        finalize(h - 1);
      }
      const int nvalid = p.N - kb * kKB;         // keys of the block inside the grid (all of them but in the last)
      if (kb == 0) m_run = -INFINITY;
      uint32_t r[2][32], pk[2][16];
      // P against the running reference, formed while the block's maximum is taken
      const float mx = logits(st, b, nvalid, m_run == -INFINITY ? 0.f : m_run, r, pk);
      // probe the next block's S and bias barriers now; the results are used at its start
      {
        const int bn = b + 1 == kSBuf ? 0 : b + 1, stn = st + 1 == kStages ? 0 : st + 1;
        const uint32_t bphn = b + 1 == kSBuf ? bph ^ 1u : bph, sphn = st + 1 == kStages ? sph ^ 1u : sph;
        probed = t + 1 < T && mbar_test_wait(&sm.s_full[g][bn], bphn) && mbar_test_wait(&sm.kv_full[stn], sphn);
      }
      // the stage's bias has been read
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.kv_empty[st]);
      // Lazy reference: it moves to the block's maximum only when that exceeds it by more than 8 (always
      // in a head's first block), so P <= 2^8 stays inside fp16 and most blocks leave the running output
      // as it is.
      const float m_new = (mx > m_run + 8.f) ? mx : m_run;
      const float ref = m_new == -INFINITY ? 0.f : m_new;
      if (m_new != m_run) {
        // the reference moved (this row only): P again, from the logits still in registers
        const float2 nref = make_float2(-ref, -ref);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 d = __fadd2_rn(make_float2(__uint_as_float(r[cc][2 * e]), __uint_as_float(r[cc][2 * e + 1])), nref);
            pk[cc][e] = pack_f16x2(ex2_approx(d.x), ex2_approx(d.y));
          }
      }
      // P over the buffer's first 32 columns, whose S is already in registers
      tmem_st16(trow + kTmS + kKB * b, pk[0]);
      tmem_st16(trow + kTmS + kKB * b + 16, pk[1]);
      // ---- the reference moved: rescale this row's running output, once the block before has been
      // added, before this block's product adds in
      if (kb != 0 && __any_sync(0xffffffffu, m_new != m_run)) {
        if (!warp_wait_bounded(&sm.pv_done[g][(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, p.w, abort_flag, 33)) { ok = false; break; }
        tc_fence_after();
        const float alpha = m_new != m_run ? ex2_approx(m_run - ref) : 1.f;
        uint32_t ro[32];
        tmem_ld32(trow + kTmPV, ro);
        const uint32_t rl = tmem_ld1(trow + kTmPV + kHd);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < kHd; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
        tmem_st32(trow + kTmPV, ro);
        tmem_st1(trow + kTmPV + kHd, __float_as_uint(__uint_as_float(rl) * alpha));
      }
      // S has been read and P stored: both go to the MMA warp
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.p_full[g][b]);
        if (g == 0 && t == 0) mbar_arrive(&sm.go1);
      }
      m_run = m_new;
      if (++kb == KB) { kb = 0; ++h; }
      if (++st == kStages) { st = 0; sph ^= 1u; }
      if (++b == kSBuf) { b = 0; bph ^= 1u; }
    }
    // the last product (every earlier one is complete with it): its own single-use barrier, since the
    // alternating ones may already be two phases on
    if (ok && warp_wait_bounded(&sm.pv_last[g], 0u, p.w, abort_flag, 34)) {
      tc_fence_after();
      finalize(3);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // a wait ran out: let copies still in flight land before the shared memory is released
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
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
    if (tid == 0) {
      // L2 prefetch of the CTA's next tile of o: its pairs' rows are one contiguous run
      const long long n0 = (t + gridDim.x) * BT;
      if (n0 < p.P) {
        const long long n1 = n0 + BT < p.P ? n0 + BT : p.P;
        prefetch_l2_bulk(p.o + n0 * kC, (uint32_t)((n1 - n0) * kC * 2));
      }
    }
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
static_assert(kTaAttSmem <= 232448, "attention shared memory");
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
  const long long grid = (long long)p.N * p.jpairs;
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
