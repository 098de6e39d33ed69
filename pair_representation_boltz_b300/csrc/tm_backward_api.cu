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
// Schedule (both precisions): recompute a, b (projection) and x (contraction, float32); the
// output backward gives dX, its transpose dX^T, and the gate's term of dzh; the two contraction
// gradients are contractions again, with other operands:
//   outgoing (X = A B^T):  dA = dX B   = incoming-form contraction of (dX^T, b)
//                          dB = dX^T A = incoming-form contraction of (dX, a)
//   incoming (X = A^T B):  dA = B dX^T = outgoing-form contraction of (b, dX)
//                          dB = A dX   = outgoing-form contraction of (a, dX^T)
// (the incoming form sums over the first index of both planes, the outgoing form over the second),
// so the forward's contraction kernels serve unchanged; the projection backward then gives dz.
// Every parameter gradient is a sum over the N^2 pairs, formed without atomics in fixed order.

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

tm_status backward_bf16(tm_ctx* c, const void* z, const float* mask, int N, bool inc, const void* dout, void* dz,
                        const tm_grads* g, cudaStream_t s, const tm_options* opt) {
  const long long P = (long long)N * N;
  const int ld = (int)align_up(N, 64);     // fp16 planes a, b, dX, dX^T: 128-byte rows
  const int ldx = (int)align_up(N, 32);    // float32 planes x (then dX, then dA), dB: 128-byte rows
  const long long tiles = (P + 127) / 128;
  const int grid = bwd_grid(tiles, c->num_sms);
  const size_t pb = align_up((size_t)kC * N * ld * 2, 256);
  const size_t xb = align_up((size_t)kC * N * ldx * 4, 256);
  const size_t zb = align_up((size_t)P * sizeof(float2), 256);
  const size_t hb = align_up((size_t)kC * P * 4, 256);
  const size_t wb = align_up((size_t)grid * 2 * kC * kC * 4, 256);
  const size_t lb = align_up((size_t)grid * 2 * kC * 4, 256);
  tm_status st = ensure_workspace(c, 4 * pb + 2 * xb + zb + hb + 3 * wb + 2 * lb + 256, s, opt);
  if (st != TM_OK) return st;
  uint8_t* q = reinterpret_cast<uint8_t*>(c->ws);
  auto take = [&](size_t n) { uint8_t* r = q; q += n; return r; };
  auto* a = reinterpret_cast<__half*>(take(pb));
  auto* b = reinterpret_cast<__half*>(take(pb));
  auto* dX = reinterpret_cast<__half*>(take(pb));
  auto* dXT = reinterpret_cast<__half*>(take(pb));
  float* x = reinterpret_cast<float*>(take(xb));     // x, then dX (float32), then dA
  float* dB = reinterpret_cast<float*>(take(xb));
  auto* zstat = reinterpret_cast<float2*>(take(zb));
  float* dzh = reinterpret_cast<float*>(take(hb));
  float* part_o = reinterpret_cast<float*>(take(wb));
  float* part_a = reinterpret_cast<float*>(take(wb));
  float* part_b = reinterpret_cast<float*>(take(wb));
  float* ln_o = reinterpret_cast<float*>(take(lb));
  float* ln_i = reinterpret_cast<float*>(take(lb));
  auto* amax = reinterpret_cast<unsigned*>(take(256));   // [0] largest |dout|, [1] largest |dX| (float bits)
  const auto* wimg = reinterpret_cast<const __half*>(c->wbwd);
  const float* ln4 = reinterpret_cast<const float*>(wimg + 6 * kC * kC);
  auto W = [&](int m) { return wimg + (size_t)m * kC * kC; };   // W_g, W_o, W_a, W_ga, W_b, W_gb
  auto SW = [&](int m) { return std::ldexp(1.0, c->bwd_wexp[m]); };

  // fp16 scales fixed by the weights: a and b (|a_c| <= the bound on |W_a zh|), zh, xh
  const double sa = pow2_scale_host(c->pv_bound[0], 14), sb = pow2_scale_host(c->pv_bound[1], 14);
  const double sz = pow2_scale_host(c->zh_bound, 14), sx = pow2_scale_host(c->xh_bound, 14);

  cudaError_t e = cudaMemsetAsync(amax, 0, 256, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemsetAsync(maxima)");
  e = timed(c, 6, P, s, [&] {
    return launch_absmax_bf16(reinterpret_cast<const __nv_bfloat16*>(dout), P * kC, amax, c->num_sms, s);
  });
  if (e != cudaSuccess) return cuda_fail(c, e, "maximum of dout launch");
  st = run_project_bf16(c, z, mask, N, zstat, a, b, ld, s, opt, true, (float)sa, (float)sb);
  if (st != TM_OK) return st;
  st = run_contract_bf16(c, a, b, N, ld, inc, 0, 0, N, N, x, ldx, X_F32, 0, s, opt, true);
  if (st != TM_OK) return st;

  BwdOutParams po{};
  po.z = reinterpret_cast<const __nv_bfloat16*>(z);
  po.zstat = zstat;
  po.x = x;
  po.ldx = ldx;
  po.xplane = (long long)N * ldx;
  po.x_unscale = (float)(1.0 / (sa * sb));
  po.dout = reinterpret_cast<const __nv_bfloat16*>(dout);
  po.amax = amax;
  po.y_bound4 = (float)(c->y_bound / 4);
  po.sz = (float)sz;
  po.sx = (float)sx;
  po.u_gg = (float)(1.0 / (SW(0) * sz));
  po.u_y = (float)(1.0 / (SW(1) * sx));
  po.u_dxh = (float)(1.0 / SW(1));
  po.u_dzh = (float)(1.0 / SW(0));
  po.u_wg = (float)(1.0 / sz);
  po.u_wo = (float)(1.0 / sx);
  po.dzh = dzh;
  po.part_w = part_o;
  po.part_ln = ln_o;
  po.w_g = W(0);
  po.w_o = W(1);
  po.ln = ln4;
  po.N = N;
  po.P = P;
  po.tiles = tiles;
  po.w = watch(c, KID_BWD_OUTPUT, opt);
  e = timed(c, 4, P, s, [&] { return launch_bwd_output_bf16(po, grid, s); });
  if (e != cudaSuccess) return cuda_fail(c, e, "output backward launch");
  e = timed(c, 6, P, s, [&] { return launch_convert_transpose(x, ldx, amax + 1, dX, dXT, N, ld, kC, s); });
  if (e != cudaSuccess) return cuda_fail(c, e, "dX conversion launch");

  float* dA = x;   // the float32 dX is dead once converted
  if (!inc) {
    st = run_contract_bf16(c, dXT, b, N, ld, true, 0, 0, N, N, dA, ldx, X_F32, 0, s, opt, true);
    if (st == TM_OK) st = run_contract_bf16(c, dX, a, N, ld, true, 0, 0, N, N, dB, ldx, X_F32, 0, s, opt, true);
  } else {
    st = run_contract_bf16(c, b, dX, N, ld, false, 0, 0, N, N, dA, ldx, X_F32, 0, s, opt, true);
    if (st == TM_OK) st = run_contract_bf16(c, a, dXT, N, ld, false, 0, 0, N, N, dB, ldx, X_F32, 0, s, opt, true);
  }
  if (st != TM_OK) return st;

  for (int side = 0; side < 2; ++side) {
    // dA = (dX sx)(b sb) / (sx sb): dV carries dX's scale (device) and its partner's (sb for dA, sa for dB).
    // |dV raw| <= N 2^14 2^14 (both fp16 operands below 2^14), so q1 = 2^(14 - 28 - ceil(log2 N)) keeps
    // dpv's fp16 values below 2^14; dpg also carries |pv| <= the bound and sigmoid' <= 1/4.
    const double sp = side == 0 ? sb : sa;
    const double raw = (double)N * 16384.0 * 16384.0;
    const double q1 = pow2_scale_host(raw, 14), q2 = pow2_scale_host(raw * c->pv_bound[side] / 4, 14);
    const double swv = SW(2 + 2 * side), swg = SW(3 + 2 * side);
    BwdProjParams pp{};
    pp.z = po.z;
    pp.zstat = zstat;
    pp.mask = mask;
    pp.dV = side == 0 ? dA : dB;
    pp.ldv = ldx;
    pp.vplane = (long long)N * ldx;
    pp.amax = amax;
    pp.sz = (float)sz;
    pp.u_pv = (float)(1.0 / (swv * sz));
    pp.u_pg = (float)(1.0 / (swg * sz));
    pp.q1 = (float)q1;
    pp.q2 = (float)q2;
    pp.u_dzh_v = (float)(1.0 / (swv * sp * q1));
    pp.u_dzh_g = (float)(1.0 / (swg * sp * q2));
    pp.u_wv = (float)(1.0 / (sp * q1 * sz));
    pp.u_wgt = (float)(1.0 / (sp * q2 * sz));
    pp.dzh = dzh;
    pp.dz = reinterpret_cast<__nv_bfloat16*>(dz);
    pp.final_pass = side;
    pp.part_w = side == 0 ? part_a : part_b;
    pp.part_ln = ln_i;
    pp.w_v = W(2 + 2 * side);
    pp.w_gt = W(3 + 2 * side);
    pp.ln = ln4;
    pp.N = N;
    pp.P = P;
    pp.tiles = tiles;
    pp.w = watch(c, KID_BWD_PROJECT, opt);
    e = timed(c, 5, P, s, [&] { return launch_bwd_project_bf16(pp, grid, s); });
    if (e != cudaSuccess) return cuda_fail(c, e, "projection backward launch");
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
    e = timed(c, 6, 0, s, [&] { return launch_sum_parts_multi(jobs, grid, s); });
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
    if (opt->block || opt->x_storage || opt->residual)
      return fail(c, TM_ERR_INVALID, "tm_backward takes no block, x_storage or residual option");
    if (opt->timeout_ms < 0) return fail(c, TM_ERR_INVALID, "negative option");
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
