// tm_backward_api.cu -- host side of the backward pass of the triangle multiplicative update
// (tm_backward in include/tm.h): the workspace of each precision and the schedule of its kernels.
#include <algorithm>
#include <cmath>

#include "tm_internal.h"

using namespace tmk;
using namespace tmh;

namespace {

// ---------------------------------------------------------------------- backward pass
//
// Schedule: recompute a, b (projection) and x (contraction, float32); the output backward gives dX
// and the gate's term of dzh; the two contraction gradients are contractions again, with other operands:
//   outgoing (X = A B^T):  dA = dX B   : x_ik = sum_j dX_ij b_jk   (mixed form: dX along j, b along k)
//                          dB = dX^T A : x_jk = sum_i dX_ij a_ik   (incoming form)
//   incoming (X = A^T B):  dA = B dX^T : x_ki = sum_j b_kj dX_ij   (outgoing form)
//                          dB = A dX   : x_kj = sum_i a_ki dX_ij   (mixed form)
// and the projection backward then gives dz. Every parameter gradient is a sum over the N^2 pairs,
// formed without atomics in fixed order.

tm_status backward_f32(tm_ctx* c, const float* z, const float* mask, int N, bool inc, const float* dout, float* dz,
                       const tm_grads* g, cudaStream_t s, const tm_options* opt) {
  const int Cz = c->c_z, Ch = c->c_h;
  const long long P = (long long)N * N;
  const int ld = N;
  const size_t plane = align_up((size_t)Ch * N * ld * 4, 256);
  const size_t vh = align_up((size_t)Ch * P * 4, 256), vz = align_up((size_t)Cz * P * 4, 256);
  const size_t part = align_up((size_t)outer_sum_splits(P) * 256 * 256 * 4, 256);
  // planes a, b, x (then dA), dX, dX^T, dB; vectors: 7 of c_h, 6 of c_z
  const size_t need = 6 * plane + 7 * vh + 6 * vz + part;
  tm_status st = ensure_workspace(c, need, s, opt);
  if (st != TM_OK) return st;
  uint8_t* q = reinterpret_cast<uint8_t*>(c->ws);
  auto take = [&](size_t n) { float* r = reinterpret_cast<float*>(q); q += n; return r; };
  float *a = take(plane), *b = take(plane), *x = take(plane), *dX = take(plane), *dXT = take(plane),
        *dB = take(plane);
  BwdF32Vectors v{};
  v.dX = dX;
  v.dXT = dXT;
  v.dA = x;            // x is dead once the output backward has run
  v.dB = dB;
  v.ld = ld;
  v.xh = take(vh);
  v.q_out_n = take(vh);
  v.q_out = take(vh);
  v.dpa = take(vh);
  v.dga = take(vh);
  v.dpb = take(vh);
  v.dgb = take(vh);
  v.dzh = take(vz);
  v.zh = take(vz);
  v.dy = take(vz);
  v.dgg = take(vz);
  v.q_in_n = take(vz);
  v.q_in = take(vz);
  float* partial = take(part);
  const F32Weights& w = c->f32w;
  cudaError_t e;
#define TM_F32_STEP(what, call)                                         \
  e = timed(c, 3, P, s, [&] { return call; });                          \
  if (e != cudaSuccess) return cuda_fail(c, e, what);
  TM_F32_STEP("projection (f32) launch", launch_project_f32(z, mask, w, a, b, N, ld, s))
  TM_F32_STEP("contraction (f32) launch",
              launch_contract_f32(inc, a, b, N, ld, Ch, 0, 0, N, N, x, ld, (long long)N * ld, s))
  TM_F32_STEP("output backward (f32) launch", launch_bwd_output_f32(x, ld, z, dout, w, N, v, s))
  float* dA = x;
  if (!inc) {
    TM_F32_STEP("dA contraction (f32) launch",
                launch_contract_f32(true, dXT, b, N, ld, Ch, 0, 0, N, N, dA, ld, (long long)N * ld, s))
    TM_F32_STEP("dB contraction (f32) launch",
                launch_contract_f32(true, dX, a, N, ld, Ch, 0, 0, N, N, dB, ld, (long long)N * ld, s))
  } else {
    TM_F32_STEP("dA contraction (f32) launch",
                launch_contract_f32(false, b, dX, N, ld, Ch, 0, 0, N, N, dA, ld, (long long)N * ld, s))
    TM_F32_STEP("dB contraction (f32) launch",
                launch_contract_f32(false, a, dXT, N, ld, Ch, 0, 0, N, N, dB, ld, (long long)N * ld, s))
  }
  TM_F32_STEP("projection backward (f32) launch", launch_bwd_project_f32(z, mask, w, N, v, dz, s))
  if (g) {
    struct Sum { float* out; const float* U; const float* V; int O, K; };
    const Sum sums[10] = {{g->w_g, v.dgg, v.zh, Cz, Cz},       {g->w_o, v.dy, v.xh, Cz, Ch},
                          {g->w_a, v.dpa, v.zh, Ch, Cz},       {g->w_ga, v.dga, v.zh, Ch, Cz},
                          {g->w_b, v.dpb, v.zh, Ch, Cz},       {g->w_gb, v.dgb, v.zh, Ch, Cz},
                          {g->ln_out_gamma, v.q_out_n, nullptr, Ch, 1}, {g->ln_out_beta, v.q_out, nullptr, Ch, 1},
                          {g->ln_in_gamma, v.q_in_n, nullptr, Cz, 1},   {g->ln_in_beta, v.q_in, nullptr, Cz, 1}};
    for (const Sum& t : sums) {
      if (!t.out) continue;
      TM_F32_STEP("parameter gradient (f32) launch", launch_outer_sum_f32(t.U, t.V, t.O, t.K, P, partial, t.out, s))
    }
  }
#undef TM_F32_STEP
  return TM_OK;
}

// Workspace of the bf16 backward with square blocks of edge B (B >= N: the whole grid at once).
struct BwdLayout {
  int N, B, rows, ld, ldxB, ldxN, grid;
  size_t plane16, xblk, vrow, hrow, zst, wpart, lpart, total;
};
BwdLayout bwd_layout(const tm_ctx* c, int N, int B) {
  BwdLayout L{};
  L.N = N;
  L.B = std::min(B, N);
  L.rows = (N + L.B - 1) / L.B;
  L.ld = (int)align_up(N, 64);      // fp16 planes a, b, dX: 128-byte rows
  L.ldxN = (int)align_up(N, 32);    // float32 row blocks of dA, dB: 128-byte rows
  L.ldxB = (int)align_up(L.B, 32);  // float32 x blocks
  L.grid = c->num_sms;
  L.plane16 = align_up((size_t)kC * N * L.ld * 2, 256);
  L.vrow = align_up((size_t)kC * L.B * L.ldxN * 4, 256);
  // one block: x shares dA's buffer (x is dead once the output backward has read it)
  L.xblk = L.rows == 1 ? 0 : align_up((size_t)kC * L.B * L.ldxB * 4, 256);
  L.hrow = align_up((size_t)kC * L.B * N * 4, 256);
  L.zst = align_up((size_t)N * N * sizeof(float2), 256);
  L.wpart = align_up((size_t)L.grid * 2 * kC * kC * 4, 256);
  L.lpart = align_up((size_t)L.grid * 2 * kC * 4, 256);
  L.total = 3 * L.plane16 + L.xblk + 2 * L.vrow + L.hrow + L.zst + 3 * L.wpart + 2 * L.lpart + 256;
  return L;
}

// The block edge: opt->block when given, else the whole grid while its workspace stays within the cap
// (the workspace limit, or 100 GB), else the largest of a few edges whose blocked workspace does.
int bwd_block(const tm_ctx* c, int N, const tm_options* opt) {
  if (opt && opt->block > 0) return opt->block;
  const size_t lim = limit_of(c, opt);
  const size_t cap = lim ? lim : (size_t)100 << 30;
  if (bwd_layout(c, N, N).total <= cap) return N;
  for (int B : {2560, 2048, 1536, 1024, 512, 256})
    if (B < N && bwd_layout(c, N, B).total <= cap) return B;
  return 256;
}

tm_status backward_bf16(tm_ctx* c, const void* z, const float* mask, int N, bool inc, const void* dout, void* dz,
                        const tm_grads* g, cudaStream_t s, const tm_options* opt) {
  const long long P = (long long)N * N;
  const int Bq = bwd_block(c, N, opt);
  if (Bq < N && (Bq < 128 || Bq % 8))
    return fail(c, TM_ERR_INVALID, "backward block edge %d: at least 128 and a multiple of 8", Bq);
  const BwdLayout L = bwd_layout(c, N, Bq);
  const int B = L.B, ld = L.ld;
  tm_status st = ensure_workspace(c, L.total, s, opt);
  if (st != TM_OK) return st;
  uint8_t* q = reinterpret_cast<uint8_t*>(c->ws);
  auto take = [&](size_t n) { uint8_t* r = q; q += n; return r; };
  auto* a = reinterpret_cast<__half*>(take(L.plane16));
  auto* b = reinterpret_cast<__half*>(take(L.plane16));
  auto* dX = reinterpret_cast<__half*>(take(L.plane16));    // fp16 dL/dx times its bound's scale
  float* dA = reinterpret_cast<float*>(take(L.vrow));       // [128][B][ldxN] rows of a block row
  float* dB = reinterpret_cast<float*>(take(L.vrow));
  float* xb = L.rows == 1 ? dA : reinterpret_cast<float*>(take(L.xblk));   // [128][B][ldxB]
  float* dzh = reinterpret_cast<float*>(take(L.hrow));      // [128][B N] of a block row
  auto* zstat = reinterpret_cast<float2*>(take(L.zst));
  float* part_o = reinterpret_cast<float*>(take(L.wpart));
  float* part_a = reinterpret_cast<float*>(take(L.wpart));
  float* part_b = reinterpret_cast<float*>(take(L.wpart));
  float* ln_o = reinterpret_cast<float*>(take(L.lpart));
  float* ln_i = reinterpret_cast<float*>(take(L.lpart));
  auto* amax = reinterpret_cast<unsigned*>(take(256));   // [0] largest |dout|, [1] bound on |dX| (float bits)
  const auto* wimg = reinterpret_cast<const __half*>(c->wbwd);
  const float* ln4 = reinterpret_cast<const float*>(wimg + 6 * kC * kC);
  auto W = [&](int m) { return wimg + (size_t)m * kC * kC; };   // W_g, W_o, W_a, W_ga, W_b, W_gb
  auto SW = [&](int m) { return std::ldexp(1.0, c->bwd_wexp[m]); };

  // fp16 scales fixed by the weights: a and b (|a_c| <= the bound on |W_a zh|), zh, xh
  const double sa = pow2_scale_host(c->pv_bound[0], 14), sb = pow2_scale_host(c->pv_bound[1], 14);
  const double sz = pow2_scale_host(c->zh_bound, 14), sx = pow2_scale_host(c->xh_bound, 14);

  // the partial sums are added to by every launch
  cudaError_t e = cudaMemsetAsync(part_o, 0, 3 * L.wpart + 2 * L.lpart + 256, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemsetAsync(partial sums)");
  e = timed(c, 6, P, s, [&] {
    return launch_absmax_bf16(reinterpret_cast<const __nv_bfloat16*>(dout), P * kC, amax, c->num_sms, s);
  });
  if (e != cudaSuccess) return cuda_fail(c, e, "maximum of dout launch");
  st = run_project_bf16(c, z, mask, N, zstat, a, b, ld, s, opt, true, (float)sa, (float)sb);
  if (st != TM_OK) return st;

  BwdOutParams po{};
  po.z = reinterpret_cast<const __nv_bfloat16*>(z);
  po.zstat = zstat;
  po.x = xb;
  po.x_unscale = (float)(1.0 / (sa * sb));
  po.dout = reinterpret_cast<const __nv_bfloat16*>(dout);
  po.amax = amax;
  po.dx_bound = (float)c->dx_bound;
  po.y_bound4 = (float)(c->y_bound / 4);
  po.sz = (float)sz;
  po.sx = (float)sx;
  po.u_gg = (float)(1.0 / (SW(0) * sz));
  po.u_y = (float)(1.0 / (SW(1) * sx));
  po.u_dxh = (float)(1.0 / SW(1));
  po.u_dzh = (float)(1.0 / SW(0));
  po.u_wg = (float)(1.0 / sz);
  po.u_wo = (float)(1.0 / sx);
  po.ldd = ld;
  po.dxplane = (long long)N * ld;
  po.part_ln = ln_o;
  po.w_g = W(0);
  po.w_o = W(1);
  po.ln = ln4;
  po.N = N;
  po.w = watch(c, KID_BWD_OUTPUT, opt);
  // x of one block (float32, the contraction of the fp16 a and b), then the output backward over it
  auto out_block = [&](int i0, int j0, int bi, int bj, bool dx_and_parts, bool with_dzh, int r0) -> tm_status {
    tm_status t = run_contract_bf16(c, a, b, N, ld, inc ? CONTRACT_IN : CONTRACT_OUT, i0, j0, bi, bj, xb,
                                    L.ldxB, X_F32, 0, s, opt, true);
    if (t != TM_OK) return t;
    BwdOutParams pb = po;
    pb.ldx = L.ldxB;
    pb.xplane = (long long)bi * L.ldxB;
    pb.i0 = i0;
    pb.j0 = j0;
    pb.bi = bi;
    pb.bj = bj;
    pb.tiles = ((long long)bi * bj + 127) / 128;
    pb.dx16 = dx_and_parts ? dX : nullptr;
    pb.part_w = dx_and_parts ? part_o : nullptr;
    pb.dzh = with_dzh ? dzh : nullptr;
    pb.dzh_P = (long long)B * N;
    pb.dzh_off = (long long)r0 * N;
    const cudaError_t ee = timed(c, 4, (long long)bi * bj, s,
                                 [&] { return launch_bwd_output_bf16(pb, bwd_grid(pb.tiles, L.grid), s); });
    return ee == cudaSuccess ? TM_OK : cuda_fail(c, ee, "output backward launch");
  };

  // blocks: first dX over the whole grid (it enters every row's contractions), then row by row
  if (L.rows > 1)
    for (int i0 = 0; i0 < N; i0 += B)
      for (int j0 = 0; j0 < N; j0 += B)
        if ((st = out_block(i0, j0, std::min(B, N - i0), std::min(B, N - j0), true, false, 0)) != TM_OK) return st;

  for (int r0 = 0; r0 < N; r0 += B) {
    const int rb = std::min(B, N - r0);
    // the gate's term of dzh for the pairs of rows [r0, r0 + rb) (one block: with dX and the sums)
    if (L.rows == 1) {
      if ((st = out_block(0, 0, N, N, true, true, 0)) != TM_OK) return st;
    } else {
      for (int j0 = 0; j0 < N; j0 += B)
        if ((st = out_block(r0, j0, rb, std::min(B, N - j0), false, true, r0)) != TM_OK) return st;
    }
    for (int side = 0; side < 2; ++side) {
      // dA or dB of the rows, float32 [128][rb][ldxN]; each carries dX's scale and its partner's
      float* dV = side == 0 ? dA : dB;
      const void *ca, *cb;
      int mode;
      if (!inc) {
        ca = dX;
        cb = side == 0 ? (const void*)b : (const void*)a;
        mode = side == 0 ? CONTRACT_MIXED : CONTRACT_IN;
      } else {
        ca = side == 0 ? (const void*)b : (const void*)a;
        cb = dX;
        mode = side == 0 ? CONTRACT_OUT : CONTRACT_MIXED;
      }
      st = run_contract_bf16(c, ca, cb, N, ld, mode, r0, 0, rb, N, dV, L.ldxN, X_F32, 0, s, opt, true);
      if (st != TM_OK) return st;
      // dV = (dX sdx)(partner s) / (sdx s) with |dX sdx| <= (largest |dX|) sdx and |partner s| < 2^14, so
      // |dV raw| <= N 2^14 (largest |dX|) sdx: the kernel takes the powers of two q1 (for dpv) and q2 (dpg,
      // which also carries |pv| <= the bound and sigmoid' <= 1/4) from that bound
      const double sp = side == 0 ? sb : sa;
      const double swv = SW(2 + 2 * side), swg = SW(3 + 2 * side);
      BwdProjParams pp{};
      pp.z = po.z;
      pp.zstat = zstat;
      pp.mask = mask;
      pp.dV = dV;
      pp.ldv = L.ldxN;
      pp.vplane = (long long)rb * L.ldxN;
      pp.amax = amax;
      pp.sz = (float)sz;
      pp.u_pv = (float)(1.0 / (swv * sz));
      pp.u_pg = (float)(1.0 / (swg * sz));
      pp.q_raw = (float)((double)N * 16384.0);
      pp.q2f = (float)(c->pv_bound[side] / 4);
      pp.u_dzh_v = (float)(1.0 / (swv * sp));
      pp.u_dzh_g = (float)(1.0 / (swg * sp));
      pp.u_wv = (float)(1.0 / (sp * sz));
      pp.u_wgt = (float)(1.0 / (sp * sz));
      pp.dzh = dzh;
      pp.dzh_P = (long long)B * N;
      pp.dzh_off = (long long)r0 * N;
      pp.dz = reinterpret_cast<__nv_bfloat16*>(dz);
      pp.final_pass = side;
      pp.part_w = side == 0 ? part_a : part_b;
      pp.part_ln = ln_i;
      pp.w_v = W(2 + 2 * side);
      pp.w_gt = W(3 + 2 * side);
      pp.ln = ln4;
      pp.N = N;
      pp.i_off = r0;
      pp.p0 = (long long)r0 * N;
      pp.P = (long long)rb * N;
      pp.tiles = (pp.P + 127) / 128;
      pp.w = watch(c, KID_BWD_PROJECT, opt);
      e = timed(c, 5, pp.P, s, [&] { return launch_bwd_project_bf16(pp, bwd_grid(pp.tiles, L.grid), s); });
      if (e != cudaSuccess) return cuda_fail(c, e, "projection backward launch");
    }
  }
  if (g) {
    struct Sum { float* out; const float* part; long long E, stride; };
    const long long WW = (long long)kC * kC;
    const Sum sums[10] = {{g->w_g, part_o, WW, 2 * WW},       {g->w_o, part_o + WW, WW, 2 * WW},
                          {g->w_a, part_a, WW, 2 * WW},       {g->w_ga, part_a + WW, WW, 2 * WW},
                          {g->w_b, part_b, WW, 2 * WW},       {g->w_gb, part_b + WW, WW, 2 * WW},
                          {g->ln_out_gamma, ln_o, kC, 2 * kC}, {g->ln_out_beta, ln_o + kC, kC, 2 * kC},
                          {g->ln_in_gamma, ln_i, kC, 2 * kC},  {g->ln_in_beta, ln_i + kC, kC, 2 * kC}};
    SumJobs jobs{};
    for (const Sum& t : sums) {
      jobs.part[jobs.n] = t.part;
      jobs.out[jobs.n] = t.out;
      jobs.E[jobs.n] = t.E;
      jobs.stride[jobs.n] = t.stride;
      ++jobs.n;
    }
    e = timed(c, 6, 0, s, [&] { return launch_sum_parts_multi(jobs, L.grid, s); });
    if (e != cudaSuccess) return cuda_fail(c, e, "parameter gradient sum launch");
  }
  return TM_OK;
}

}  // namespace

extern "C" {

tm_status tm_backward(tm_ctx* c, const void* z, const float* mask, int N, tm_dtype dtype, tm_direction dir,
                      const void* dout, void* dz, const tm_grads* grads, void* stream, const tm_options* opt) {
  tm_status st = check_common(c, N, dtype);
  if (st != TM_OK) return st;
  if (dir != TM_OUTGOING && dir != TM_INCOMING) return fail(c, TM_ERR_INVALID, "unknown direction %d", (int)dir);
  if (!z || !dout || !dz || !aligned16(z) || !aligned16(dout) || !aligned16(dz))
    return fail(c, TM_ERR_INVALID, "z, dout and dz must be non-null and 16-byte aligned");
  if (mask && (reinterpret_cast<uintptr_t>(mask) & 3u)) return fail(c, TM_ERR_INVALID, "mask must be 4-byte aligned");
  if (opt) {
    for (int r : opt->reserved)
      if (r) return fail(c, TM_ERR_INVALID, "tm_options.reserved must be zero");
    if (opt->x_storage || opt->residual) return fail(c, TM_ERR_INVALID, "tm_backward takes no x_storage or residual option");
    if (opt->timeout_ms < 0 || opt->block < 0) return fail(c, TM_ERR_INVALID, "negative option");
    if (opt->block && dtype != TM_BF16) return fail(c, TM_ERR_INVALID, "the float32 backward takes no block option");
  }
  if (grads) {
    const float* gp[10] = {grads->ln_in_gamma, grads->ln_in_beta, grads->w_a, grads->w_ga, grads->w_b,
                           grads->w_gb, grads->w_g, grads->ln_out_gamma, grads->ln_out_beta, grads->w_o};
    for (const float* q : gp)
      if (q && (reinterpret_cast<uintptr_t>(q) & 15u))
        return fail(c, TM_ERR_INVALID, "gradient arrays must be 16-byte aligned");
  }
  const size_t zbytes = (size_t)N * N * c->c_z * (dtype == TM_BF16 ? 2 : 4);
  if (ranges_overlap(z, zbytes, dz, zbytes)) return fail(c, TM_ERR_INVALID, "dz overlaps z");
  if (dz != dout && ranges_overlap(dout, zbytes, dz, zbytes))
    return fail(c, TM_ERR_INVALID, "dz overlaps dout without being dout");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool inc = dir == TM_INCOMING;
  if (dtype == TM_F32)
    return backward_f32(c, reinterpret_cast<const float*>(z), mask, N, inc, reinterpret_cast<const float*>(dout),
                        reinterpret_cast<float*>(dz), grads, s, opt);
  return backward_bf16(c, z, mask, N, inc, dout, dz, grads, s, opt);
}

}  // extern "C"
