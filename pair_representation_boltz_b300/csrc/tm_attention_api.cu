// tm_attention_api.cu -- host side of triangle attention (tm_attn_create, tm_attn_forward in
// include/tm.h): the layer's weight images, argument checks, the workspace, the tensor maps and the
// three launches.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "tm_internal.h"

using namespace tmk;
using namespace tmh;

extern "C" {

tm_status tm_attn_create(int c_z, int heads, int c_head, const tm_attn_weights* w, tm_ctx** out_ctx) {
  if (!w || !out_ctx) return TM_ERR_INVALID;
  const float* req[] = {w->ln_gamma, w->ln_beta, w->w_q, w->w_k, w->w_v, w->w_b, w->w_g, w->w_o};
  for (const float* q : req)
    if (!q) return TM_ERR_INVALID;
  if (c_z < 1 || heads < 1 || c_head < 1) return TM_ERR_INVALID;
  if (c_z != kC || heads != 4 || c_head != 32) return TM_ERR_UNSUPPORTED;
  tm_ctx* c = new tm_ctx();
  c->layer = 1;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) {
    delete c;
    cudaGetLastError();
    return TM_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  c->c_z = c_z;
  c->c_h = heads * c_head;
  if (const char* env = std::getenv("TM_WORKSPACE_LIMIT")) c->env_limit = (size_t)std::strtoull(env, nullptr, 10);
  e = cudaHostAlloc(reinterpret_cast<void**>(&c->status_h), 64, cudaHostAllocMapped);
  if (e != cudaSuccess) {
    tm_destroy(c);
    cudaGetLastError();
    return TM_ERR_CUDA;
  }
  std::memset(c->status_h, 0, 64);
  cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->status_d), c->status_h, 0);
  // Every intermediate of the path is stored as fp16 (normal values 2^-14 .. 65504). The weights bound
  // each one for any input: with zh = gamma (z - mu) rstd + beta and ||(z - mu) rstd|| <= sqrt(c_z),
  // |zh_k| <= sqrt(c_z) |gamma_k| + |beta_k| and |(W zh)_c| <= sqrt(c_z) ||W[c] diag(gamma)|| + |(W beta)_c|.
  // zh and v are stored times powers of two 2^sz, 2^sv that put those bounds near 2^14 (o, a gated
  // average of v, shares v's); the products undo the scales in their epilogues, exactly. q (which
  // carries log2(e)/sqrt(c)), k and the bias (times log2(e)) set the logits, whose error is absolute,
  // and are stored unscaled: weights that could push them past 2^15 are refused.
  const double kLog2e = 1.4426950408889634, kQ = kLog2e / std::sqrt(32.0);
  int sz = 0, sv = 0;
  {
    double zb = 0;
    for (int k = 0; k < kC; ++k) zb = std::max(zb, std::sqrt((double)kC) * std::fabs((double)w->ln_gamma[k]) +
                                                       std::fabs((double)w->ln_beta[k]));
    auto bound = [&](const float* W, int rows) {
      double mx = 0;
      for (int r = 0; r < rows; ++r) {
        double n2 = 0, b = 0;
        for (int k = 0; k < kC; ++k) {
          const double v = (double)W[(size_t)r * kC + k];
          n2 += v * v * (double)w->ln_gamma[k] * (double)w->ln_gamma[k];
          b += v * (double)w->ln_beta[k];
        }
        mx = std::max(mx, std::sqrt((double)kC * n2) + std::fabs(b));
      }
      return mx;
    };
    const double lim = 32768.0;
    const double bq = kQ * bound(w->w_q, kC), bk = bound(w->w_k, kC), bv = bound(w->w_v, kC),
                 bb = kLog2e * bound(w->w_b, 4);
    if (!(bq < lim && bk < lim && bb < lim) || !std::isfinite(zb) || !std::isfinite(bv)) {
      tm_destroy(c);
      return TM_ERR_UNSUPPORTED;
    }
    auto expo = [](double b) { return b > 0 ? std::min(60, std::max(-60, 14 - (int)std::ceil(std::log2(b)))) : 0; };
    sz = expo(zb);
    sv = expo(bv);
  }
  const size_t T = (size_t)kC * kC;
  std::vector<__half> img(5 * T);
  const float* mats[5] = {w->w_q, w->w_k, w->w_v, w->w_g, w->w_o};
  for (int m = 0; m < 5; ++m) {
    const int ex = fp16_image_exponent(mats[m]);
    make_tile_image_h(mats[m], std::ldexp(1.0, ex), img.data() + m * T);
    if (m < 4) {
      const double sc = std::ldexp(1.0, -ex - sz + (m == 2 ? sv : 0));
      c->ta_wscale[m] = (float)(m == 0 ? sc * kQ : sc);
    } else {
      c->ta_oscale = (float)std::ldexp(1.0, -ex - sv);
    }
  }
  c->ta_bscale = (float)(kLog2e * std::ldexp(1.0, -sz));
  std::vector<float> f(2 * kC + 4 * kC);
  for (int k = 0; k < kC; ++k) {
    f[k] = (float)std::ldexp((double)w->ln_gamma[k], sz);
    f[kC + k] = (float)std::ldexp((double)w->ln_beta[k], sz);
  }
  for (int k = 0; k < 4 * kC; ++k) f[2 * kC + k] = w->w_b[k];
  const size_t ib = img.size() * sizeof(img[0]);
  e = cudaMalloc(&c->ta_w, ib + f.size() * sizeof(float));
  if (e == cudaSuccess) e = cudaMemcpy(c->ta_w, img.data(), ib, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(reinterpret_cast<uint8_t*>(c->ta_w) + ib, f.data(), f.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    tm_destroy(c);
    cudaGetLastError();
    return TM_ERR_CUDA;
  }
  *out_ctx = c;
  return TM_OK;
}

tm_status tm_attn_forward(tm_ctx* c, const void* z, const float* mask, int N, tm_dtype dtype, tm_attn_node node,
                          void* out, void* stream, const tm_options* opt) {
  if (!c) return TM_ERR_INVALID;
  c->err.clear();
  if (c->layer != 1) return fail(c, TM_ERR_INVALID, "this ctx holds a triangle multiplicative update (tm_forward)");
  if (N < 1 || N > 65535) return fail(c, TM_ERR_INVALID, "N=%d outside [1, 65535]", N);
  if (dtype != TM_BF16) return fail(c, dtype == TM_F32 ? TM_ERR_UNSUPPORTED : TM_ERR_INVALID, "triangle attention runs in bf16");
  if (node != TM_ATTN_STARTING && node != TM_ATTN_ENDING) return fail(c, TM_ERR_INVALID, "unknown node %d", (int)node);
  if (!z || !out || !aligned16(z) || !aligned16(out))
    return fail(c, TM_ERR_INVALID, "z and out must be non-null and 16-byte aligned");
  if (mask && (reinterpret_cast<uintptr_t>(mask) & 3u)) return fail(c, TM_ERR_INVALID, "mask must be 4-byte aligned");
  if (opt) {
    for (int r : opt->reserved)
      if (r) return fail(c, TM_ERR_INVALID, "tm_options.reserved must be zero");
    if (opt->block || opt->x_storage || opt->residual || opt->timeout_ms < 0)
      return fail(c, TM_ERR_INVALID, "tm_attn_forward takes only timeout_ms and workspace_limit");
  }
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != c->device) return fail(c, TM_ERR_INVALID, "current device %d is not the ctx's device %d", dev, c->device);
  tm_status st = check_device_status(c);
  if (st != TM_OK) return st;
  const size_t zbytes = (size_t)N * N * kC * 2;
  if (ranges_overlap(z, zbytes, out, zbytes)) return fail(c, TM_ERR_INVALID, "out overlaps z");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool tr = node == TM_ATTN_ENDING;
  const long long P = (long long)N * N;
  const long long ldv = (long long)align_up(N, 64), ldb = ldv;
  const size_t pb = align_up(zbytes, 256);
  const size_t vb = align_up((size_t)N * kC * ldv * 2, 256);
  const size_t bb = align_up((size_t)4 * N * ldb * 2, 256);
  st = ensure_workspace(c, 4 * pb + vb + bb, s, opt);
  if (st != TM_OK) return st;
  uint8_t* q8 = reinterpret_cast<uint8_t*>(c->ws);
  auto* q = reinterpret_cast<__half*>(q8);
  auto* k = reinterpret_cast<__half*>(q8 + pb);
  auto* g = reinterpret_cast<__half*>(q8 + 2 * pb);
  auto* o = reinterpret_cast<__half*>(q8 + 3 * pb);
  auto* vt = reinterpret_cast<__half*>(q8 + 4 * pb);
  auto* bias = reinterpret_cast<__half*>(q8 + 4 * pb + vb);
  const auto* wimg = reinterpret_cast<const __half*>(c->ta_w);
  const float* wf = reinterpret_cast<const float*>(wimg + 5 * kC * kC);
  const long long tiles = (P + 127) / 128;
  const int grid = (int)std::min<long long>(tiles, c->num_sms);

  TaProjectParams pp{};
  pp.z = reinterpret_cast<const __nv_bfloat16*>(z);
  pp.mask = mask;
  pp.transpose = tr ? 1 : 0;
  pp.ln = wf;
  pp.w_b = wf + 2 * kC;
  pp.w_q = wimg;
  pp.w_k = wimg + kC * kC;
  pp.w_v = wimg + 2 * kC * kC;
  pp.w_g = wimg + 3 * kC * kC;
  for (int m = 0; m < 4; ++m) pp.wscale[m] = c->ta_wscale[m];
  pp.bscale = c->ta_bscale;
  pp.q = q;
  pp.k = k;
  pp.g = g;
  pp.vt = vt;
  pp.b = bias;
  pp.ldv = ldv;
  pp.ldb = ldb;
  pp.N = N;
  pp.P = P;
  pp.tiles = tiles;
  pp.w = watch(c, KID_TA_PROJECT, opt);
  cudaError_t e = timed(c, 8, P, s, [&] { return launch_ta_project(pp, grid, s); });
  if (e != cudaSuccess) return cuda_fail(c, e, "attention projection launch");

  CUtensorMap qmap, kmap, vmap, bmap;
  {
    const cuuint64_t d[3] = {(cuuint64_t)kC, (cuuint64_t)N, (cuuint64_t)N};
    const cuuint64_t st2[2] = {(cuuint64_t)kC * 2, (cuuint64_t)N * kC * 2};
    if (!encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, q, d, st2, kBoxTaQK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, k, d, st2, kBoxTaK, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (q/k)");
    const cuuint64_t dv[3] = {(cuuint64_t)N, (cuuint64_t)kC, (cuuint64_t)N};
    const cuuint64_t sv[2] = {(cuuint64_t)ldv * 2, (cuuint64_t)kC * ldv * 2};
    if (!encode(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vt, dv, sv, kBoxTaV, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (v)");
    const cuuint64_t db[3] = {(cuuint64_t)N, (cuuint64_t)N, 4};
    const cuuint64_t sb[2] = {(cuuint64_t)ldb * 2, (cuuint64_t)N * ldb * 2};
    if (!encode(&bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, bias, db, sb, kBoxTaBias, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (bias)");
  }
  TaAttendParams pa{};
  pa.mask = mask;
  pa.g = g;
  pa.o = o;
  pa.N = N;
  pa.jpairs = ((N + 127) / 128 + 1) / 2;
  pa.w = watch(c, KID_TA_ATTEND, opt);
  e = timed(c, 9, P, s, [&] { return launch_ta_attend(qmap, kmap, vmap, bmap, pa, s); });
  if (e != cudaSuccess) return cuda_fail(c, e, "attention launch");

  TaOutParams po{};
  po.o = o;
  po.w_o = wimg + 4 * kC * kC;
  po.oscale = c->ta_oscale;
  po.out = reinterpret_cast<__nv_bfloat16*>(out);
  po.transpose = tr ? 1 : 0;
  po.N = N;
  po.P = P;
  po.tiles = tiles;
  po.w = watch(c, KID_TA_OUT, opt);
  e = timed(c, 10, P, s, [&] { return launch_ta_out(po, grid, s); });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "attention output launch");
}

}  // extern "C"
