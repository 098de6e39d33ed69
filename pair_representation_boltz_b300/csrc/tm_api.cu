// tm_api.cu -- the C ABI of libtm (declared in include/tm.h): argument
// checking, weight preparation, the workspace, TMA tensor maps and the
// block-streamed schedule of the triangle multiplicative update. The backward
// pass's host side is in tm_backward_api.cu, triangle attention's in
// tm_attention_api.cu; what they share with this file is in tm_internal.h.
//
// Schedule of one bf16 update (tm_forward):
//   projection       z -> a, b                    (one launch, whole grid)
//   for each output block (I, J) of the B x B block grid:
//     contraction    a, b -> x block (float32)    (one launch)
//     finish         x block, z -> out block      (one launch)
// Only one float32 x block is alive at a time, so for N = 10000 and
// B = 2500 the device holds z, a, b and out plus a 3.2 GB x block. The 2D
// block tiling of the pair representation is the one the pages use across
// GPUs ("2D tiling da pair representation" section of "NVIDIA BioNeMo escala
// modelagem biomolecular com context parallelism e quebra barreira de memória
// da GPU"), and streaming the blocks replaces the in-model chunking that the
// "O problema dos workarounds atuais" section of that page describes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "tm_internal.h"

using namespace tmk;

using namespace tmk;
using namespace tmh;

namespace {
const char* kStatusText[] = {"ok", "invalid argument", "unsupported configuration", "out of workspace memory",
                             "CUDA error", "device wait timed out"};
}  // namespace

namespace tmh {

// The driver's tensor-map encoder, looked up once per process (contexts on different host threads may
// ask for it at the same time).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

tm_status fail(tm_ctx* c, tm_status s, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    c->err = buf;
  }
  return s;
}

tm_status cuda_fail(tm_ctx* c, cudaError_t e, const char* what) {
  cudaGetLastError();
  return fail(c, TM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const Box& b, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint32_t esz = dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4u : 2u;
  if (esz != b.esz || (rank == 2 && b.d2 != 1)) return false;   // the box constant must match the map
  const cuuint32_t shape[3] = {b.d0, b.d1, b.d2};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, shape, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

Watch watch(const tm_ctx* c, int kernel, const tm_options* opt) {
  Watch w;
  w.status = c->status_d;
  const int ms = (opt && opt->timeout_ms > 0) ? opt->timeout_ms : 2000;
  w.limit_ns = (unsigned long long)ms * 1000000ull;
  w.kernel = kernel;
  return w;
}

cudaEvent_t take_event(tm_ctx* c) {
  if (!c->event_pool.empty()) {
    cudaEvent_t e = c->event_pool.back();
    c->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}


tm_status check_device_status(tm_ctx* c) {
  volatile int* st = c->status_h;
  if (st[0] != 0) {
    const int code = st[0];
    c->err = "device wait timed out in kernel " + std::to_string(st[1]) + " at site " + std::to_string(st[2]) +
             " (block " + std::to_string(st[3]) + ")";
    st[0] = 0;
    return code == TM_ERR_TIMEOUT ? TM_ERR_TIMEOUT : TM_ERR_CUDA;
  }
  return TM_OK;
}

size_t limit_of(const tm_ctx* c, const tm_options* opt) {
  if (opt && opt->workspace_limit) return opt->workspace_limit;
  return c->env_limit;  // 0 = none
}

tm_status ensure_workspace(tm_ctx* c, size_t bytes, cudaStream_t s, const tm_options* opt) {
  const size_t lim = limit_of(c, opt);
  if (lim && bytes > lim)
    return fail(c, TM_ERR_OOM, "workspace of %zu bytes exceeds the limit of %zu bytes", bytes, lim);
  if (c->ws_bytes >= bytes) return TM_OK;
  if (c->ws) {
    cudaError_t e = cudaFreeAsync(c->ws, s);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaFreeAsync(workspace)");
    c->ws = nullptr;
    c->ws_bytes = 0;
  }
  cudaError_t e = cudaMallocAsync(&c->ws, bytes, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    c->ws = nullptr;
    return fail(c, TM_ERR_OOM, "cudaMallocAsync(%zu bytes): %s", bytes, cudaGetErrorString(e));
  }
  c->ws_bytes = bytes;
  c->ws_stream = s;
  return TM_OK;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// ------------------------------------------------------------------ host weight preparation
inline void split_bf16(double v, __nv_bfloat16* hi, __nv_bfloat16* lo) {
  *hi = __float2bfloat16_rn((float)v);
  *lo = __float2bfloat16_rn((float)(v - (double)__bfloat162float(*hi)));
}

// W [128][128] (row-major [out][in]) as bf16 in the 128-byte-swizzled K-major tile layout of the
// per-pair kernels (64-column halves 16 KB apart, 128-byte rows, 16-byte unit u of row r at u ^ (r % 8)).
void make_tile_image(const float* W, __nv_bfloat16* img) {
  const int C = kC;
  for (int r = 0; r < C; ++r)
    for (int k = 0; k < C; ++k) {
      const int half = k / 64, u = (k % 64) / 8, e = k % 8;
      const size_t byte = (size_t)half * (C * 64 * 2) + (size_t)r * 128 + (size_t)((u ^ (r & 7)) * 16) + e * 2;
      img[byte / 2] = __float2bfloat16_rn(W[(size_t)r * C + k]);
    }
}

// The same image in fp16, every weight multiplied by `scale` (a power of two) first.
void make_tile_image_h(const float* W, double scale, __half* img) {
  const int C = kC;
  for (int r = 0; r < C; ++r)
    for (int k = 0; k < C; ++k) {
      const int half = k / 64, u = (k % 64) / 8, e = k % 8;
      const size_t byte = (size_t)half * (C * 64 * 2) + (size_t)r * 128 + (size_t)((u ^ (r & 7)) * 16) + e * 2;
      img[byte / 2] = __float2half_rn((float)((double)W[(size_t)r * C + k] * scale));
    }
}

// Power-of-two exponent s that brings the largest |W| of a 128 x 128 matrix into [2^13, 2^14), so that
// its fp16 image keeps every entry normal down to 2^-27 of the largest.
int fp16_image_exponent(const float* W) {
  double mx = 0;
  for (int i = 0; i < kC * kC; ++i) mx = std::max(mx, std::fabs((double)W[i]));
  if (!(mx > 0)) return 0;
  return 13 - (int)std::floor(std::log2(mx));
}

tm_status prepare_tensor_core_weights(tm_ctx* c, const tm_weights* w) {
  const int C = kC;
  std::vector<__nv_bfloat16> k1(2 * 2 * 256 * C);
  std::vector<float> k1c(2 * 512);
  // Gate rows carry a factor -log2(e): the projection kernel takes sigmoid(g) = 1 / (1 + 2^(-g log2 e))
  // straight from its accumulator. Bound on |a_c| (and |b_c|) for the fp16 storage of x: with
  // W' = W diag(gamma_in), |W zh| = |rstd W'(z - mu) + W beta| <= sqrt(c_z) ||W'_c|| + |(W beta)_c|, since
  // ||z - mu|| rstd <= sqrt(c_z); the gate and the mask only shrink it.
  const double kNegLog2e = -1.4426950408889634;
  double abound[2][kC];
  for (int h = 0; h < 2; ++h) {
    const float* wp = h == 0 ? w->w_a : w->w_b;
    const float* wgt = h == 0 ? w->w_ga : w->w_gb;
    for (int n = 0; n < 256; ++n) {
      const float* src = n < C ? wp + (size_t)n * C : wgt + (size_t)(n - C) * C;
      const double f = n < C ? 1.0 : kNegLog2e;
      double rs = 0, bias = 0, norm2 = 0;
      for (int k = 0; k < C; ++k) {
        const double v = f * (double)src[k] * (double)w->ln_in_gamma[k];
        norm2 += v * v;
        __nv_bfloat16 hi, lo;
        split_bf16(v, &hi, &lo);
        k1[((size_t)(h * 2 + 0) * 256 + n) * C + k] = hi;
        k1[((size_t)(h * 2 + 1) * 256 + n) * C + k] = lo;
        rs += (double)__bfloat162float(hi) + (double)__bfloat162float(lo);
        bias += f * (double)src[k] * (double)w->ln_in_beta[k];
      }
      k1c[h * 512 + n] = (float)rs;
      k1c[h * 512 + 256 + n] = (float)bias;
      if (n < C) abound[h][n] = std::sqrt((double)C * norm2) + std::fabs(bias);
    }
  }
  c->ab_bound = 0;
  c->pv_bound[0] = c->pv_bound[1] = 0;
  for (int n = 0; n < C; ++n) {
    c->ab_bound = std::max(c->ab_bound, abound[0][n] * abound[1][n]);
    c->pv_bound[0] = std::max(c->pv_bound[0], abound[0][n]);
    c->pv_bound[1] = std::max(c->pv_bound[1], abound[1][n]);
  }
  // W_o' = W_o diag(gamma_out), scaled by 2^e into fp16's top binades
  double maxabs = 0;
  for (int o = 0; o < C; ++o)
    for (int k = 0; k < C; ++k)
      maxabs = std::max(maxabs, std::fabs((double)w->w_o[(size_t)o * C + k] * (double)w->ln_out_gamma[k]));
  int e = 0;
  if (maxabs > 0) e = 14 - (int)std::floor(std::log2(maxabs));
  const double sc = std::ldexp(1.0, e);
  std::vector<__half> wo(C * C);
  std::vector<__nv_bfloat16> wg(2 * C * C);
  std::vector<float> k3c(4 * C);
  for (int o = 0; o < C; ++o) {
    double bo = 0, rs = 0, bg = 0;
    for (int k = 0; k < C; ++k) {
      wo[(size_t)o * C + k] = __float2half_rn((float)((double)w->w_o[(size_t)o * C + k] * w->ln_out_gamma[k] * sc));
      bo += (double)w->w_o[(size_t)o * C + k] * (double)w->ln_out_beta[k];
      // the finish kernel's gate reads W_g zh / 2 (sigmoid through tanh of the half argument)
      const double vg = 0.5 * (double)w->w_g[(size_t)o * C + k] * (double)w->ln_in_gamma[k];
      __nv_bfloat16 hi, lo;
      split_bf16(vg, &hi, &lo);
      wg[(size_t)o * C + k] = hi;
      wg[(size_t)(C + o) * C + k] = lo;
      rs += (double)__bfloat162float(hi) + (double)__bfloat162float(lo);
      bg += 0.5 * (double)w->w_g[(size_t)o * C + k] * (double)w->ln_in_beta[k];
    }
    k3c[o] = (float)rs;
    k3c[C + o] = (float)bg;
    k3c[2 * C + o] = (float)(0.5 * bo);     // the output projection is read as y / 2 as well
  }
  c->inv_scale_o = (float)std::ldexp(1.0, -e - 1);
  // row sums of the stored (scaled fp16) W_o', times the scale that undoes it: the fp16-x finish
  // kernel applies LayerNorm_out after the MMA, y/2 = inv rstd (W_o' x - mu rowsum W_o') + bias/2
  for (int o = 0; o < C; ++o) {
    double rs = 0;
    for (int k = 0; k < C; ++k) rs += (double)__half2float(wo[(size_t)o * C + k]);
    k3c[3 * C + o] = (float)(rs * c->inv_scale_o);
  }
  std::memcpy(c->k3c_host, k3c.data(), sizeof c->k3c_host);

  cudaError_t err;
#define TM_UP(dst, vec)                                                                       \
  err = cudaMalloc(&dst, vec.size() * sizeof(vec[0]));                                        \
  if (err != cudaSuccess) return cuda_fail(c, err, "cudaMalloc(weights)");                    \
  err = cudaMemcpy(dst, vec.data(), vec.size() * sizeof(vec[0]), cudaMemcpyHostToDevice);     \
  if (err != cudaSuccess) return cuda_fail(c, err, "cudaMemcpy(weights)");
  TM_UP(c->wk1, k1)
  TM_UP(c->k1c, k1c)
  TM_UP(c->wo16, wo)
  TM_UP(c->wg16, wg)
#undef TM_UP
  {
    // Backward images: W [out][in] as fp16, times a power of two each, in the 128-byte-swizzled K-major
    // tile layout the backward kernels copy straight into shared memory (64-column halves 16 KB apart,
    // 128-byte rows, 16-byte unit u of row r at unit u ^ (r % 8)). Bounds for the fp16 scales of the
    // backward's per-pair operands: |zh_k| <= sqrt(c_z) |gamma_in,k| + |beta_in,k|, |xh_k| likewise
    // with the output LayerNorm, |(W_o xh)_c| <= sqrt(c_h) ||W_o[c] diag(gamma_out)|| + |(W_o beta_out)_c|.
    const float* src[6] = {w->w_g, w->w_o, w->w_a, w->w_ga, w->w_b, w->w_gb};
    std::vector<__half> img(6 * C * C);
    for (int m = 0; m < 6; ++m) {
      c->bwd_wexp[m] = fp16_image_exponent(src[m]);
      make_tile_image_h(src[m], std::ldexp(1.0, c->bwd_wexp[m]), img.data() + (size_t)m * C * C);
    }
    double zb = 0, xb = 0, yb = 0;
    for (int k = 0; k < C; ++k) {
      zb = std::max(zb, std::sqrt((double)C) * std::fabs((double)w->ln_in_gamma[k]) + std::fabs((double)w->ln_in_beta[k]));
      xb = std::max(xb, std::sqrt((double)C) * std::fabs((double)w->ln_out_gamma[k]) + std::fabs((double)w->ln_out_beta[k]));
    }
    for (int o = 0; o < C; ++o) {
      double n2 = 0, b = 0;
      for (int k = 0; k < C; ++k) {
        const double v = (double)w->w_o[(size_t)o * C + k];
        n2 += v * v * (double)w->ln_out_gamma[k] * (double)w->ln_out_gamma[k];
        b += v * (double)w->ln_out_beta[k];
      }
      yb = std::max(yb, std::sqrt((double)C * n2) + std::fabs(b));
    }
    c->zh_bound = zb;
    c->xh_bound = xb;
    c->y_bound = yb;
    // dL/dx = r_x (u - mean(u) - n mean(u n)) with u = gamma_out dxh, dxh = W_o^T (dout sigmoid(g)),
    // n = x_hat: r_x <= 1/sqrt(eps), |n_c| <= sqrt(c_h), |mean(u n)| <= max|u|, |u_c| <= |gamma_out,c|
    // ||W_o[:, c]||_1 max|dout|
    double ub = 0;
    for (int k = 0; k < C; ++k) {
      double s1 = 0;
      for (int o = 0; o < C; ++o) s1 += std::fabs((double)w->w_o[(size_t)o * C + k]);
      ub = std::max(ub, std::fabs((double)w->ln_out_gamma[k]) * s1);
    }
    c->dx_bound = (2.0 + std::sqrt((double)C)) / std::sqrt(1e-5) * ub;
    std::vector<float> ln(4 * C);
    for (int k = 0; k < C; ++k) {
      ln[k] = w->ln_in_gamma[k];
      ln[C + k] = w->ln_in_beta[k];
      ln[2 * C + k] = w->ln_out_gamma[k];
      ln[3 * C + k] = w->ln_out_beta[k];
    }
    const size_t ib = img.size() * sizeof(img[0]);
    err = cudaMalloc(&c->wbwd, ib + ln.size() * sizeof(float));
    if (err != cudaSuccess) return cuda_fail(c, err, "cudaMalloc(backward weights)");
    err = cudaMemcpy(c->wbwd, img.data(), ib, cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
      err = cudaMemcpy(reinterpret_cast<uint8_t*>(c->wbwd) + ib, ln.data(), ln.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) return cuda_fail(c, err, "cudaMemcpy(backward weights)");
  }

  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, 1024};
    const cuuint64_t str[1] = {(cuuint64_t)C * 2};
    if (!encode(&c->wk1_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->wk1, dims, str, kBoxProjW, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (projection weights)");
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)C};
    const cuuint64_t str[1] = {(cuuint64_t)C * 2};
    if (!encode(&c->wo_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, c->wo16, dims, str, kBoxFinishW, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (W_o)");
    const cuuint64_t dims2[2] = {(cuuint64_t)C, (cuuint64_t)(2 * C)};
    if (!encode(&c->wg_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->wg16, dims2, str, kBoxFinishW, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (W_g)");
  }
  return TM_OK;
}

// ------------------------------------------------------------------ bf16 stage launchers (arguments checked)
double pow2_scale_host(double bound, int target) {
  if (!(bound > 0) || !std::isfinite(bound)) return 1.0;
  int e = 0;
  std::frexp(bound, &e);   // bound = m 2^e, 0.5 <= m < 1
  const int ex = std::min(127, std::max(-126, target - e));
  return std::ldexp(1.0, ex);
}

tm_status run_project_bf16(tm_ctx* c, const void* z, const float* mask, int N, float2* zstat, void* a,
                           void* b, int ld, cudaStream_t s, const tm_options* opt, bool out_f16, float scale_a,
                           float scale_b, const float* mask_col, bool separate_col_mask) {
  CUtensorMap zmap;
  const cuuint64_t dims[3] = {(cuuint64_t)kC, (cuuint64_t)N, (cuuint64_t)N};
  const cuuint64_t str[2] = {(cuuint64_t)kC * 2, (cuuint64_t)N * kC * 2};
  if (!encode(&zmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, z, dims, str, kBoxProjZ, CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(c, TM_ERR_CUDA, "tensor map (z, projection)");
  CUtensorMap amap, bmap;
  {
    const cuuint64_t od[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)kC};
    const cuuint64_t os[2] = {(cuuint64_t)ld * 2, (cuuint64_t)N * ld * 2};
    if (!encode(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a, od, os, kBoxProjOut, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, od, os, kBoxProjOut, CU_TENSOR_MAP_SWIZZLE_64B))
      return fail(c, TM_ERR_CUDA, "tensor map (a/b, projection store)");
  }
  ProjectParams p;
  p.a = reinterpret_cast<__nv_bfloat16*>(a);
  p.b = reinterpret_cast<__nv_bfloat16*>(b);
  p.mask_col = separate_col_mask ? mask_col : mask;
  p.out_f16 = out_f16 ? 1 : 0;
  p.out_scale[0] = scale_a;
  p.out_scale[1] = scale_b;
  p.mask = mask;
  p.consts = c->k1c;
  p.zstat = zstat;
  p.N = N;
  p.ld = ld;
  p.tiles_per_row = (N + kProjTileJ - 1) / kProjTileJ;
  p.total_tiles = (long long)N * p.tiles_per_row;
  p.w = watch(c, KID_PROJECT, opt);
  cudaError_t e = timed(c, 0, (long long)N * N, s, [&] { return launch_project_bf16(zmap, c->wk1_map, amap, bmap, p, c->num_sms, s); });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "projection launch");
}

tm_status run_contract_bf16(tm_ctx* c, const void* a, const void* b, int N, int ld, int mode,
                            int i0, int j0, int bi, int bj, void* x, int ldx, XFormat xf, int x_exp,
                            cudaStream_t s, const tm_options* opt, bool ab_f16, bool accumulate) {
  CUtensorMap amap, bmap;
  const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)kC};
  const cuuint64_t str[2] = {(cuuint64_t)ld * 2, (cuuint64_t)N * ld * 2};
  // A along k (outgoing, mixed) or along i (incoming); B along k (outgoing) or along j (incoming, mixed)
  const bool a_k = mode != CONTRACT_IN, b_k = mode == CONTRACT_OUT;
  if (!encode(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a, dims, str, a_k ? kBoxContractOutA : kBoxContractIn,
              CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, dims, str, b_k ? kBoxContractOutB : kBoxContractIn,
              CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(c, TM_ERR_CUDA, "tensor map (a/b, contraction)");
  ContractParams p;
  p.x = x;
  p.ab_f16 = ab_f16 ? 1 : 0;
  p.accumulate = accumulate ? 1 : 0;
  p.x_f16 = xf == X_F16 ? 1 : 0;
  p.x_exp = x_exp;
  p.ldx = ldx;
  p.chan_stride = (long long)bi * ldx;
  p.N = N;
  p.i0 = i0;
  p.j0 = j0;
  p.bi = bi;
  p.bj = bj;
  p.i_base = i0 & ~7;
  p.j_base = j0 & ~7;
  p.tiles_i = (i0 + bi - p.i_base + kContractBM - 1) / kContractBM;
  p.tiles_j = (j0 + bj - p.j_base + kContractBN - 1) / kContractBN;
  p.total_tiles = (long long)kC * p.tiles_i * p.tiles_j;
  {
    const int rest = j0 + bj - p.j_base - (p.tiles_j - 1) * kContractBN;   // in [1, 256]
    p.last_n = (rest + 15) / 16 * 16;
  }
  // TMA stores need every box to start at a non-negative, 16-byte-aligned coordinate: block origins on the
  // 8-element grid give i_base == i0 and j_base == j0, so the tiles start at 0 in the block's own x map.
  p.tma_store = ((i0 & 7) == 0 && (j0 & 7) == 0) ? 1 : 0;
  if (accumulate && (!p.tma_store || xf != X_F32))
    return fail(c, TM_ERR_INVALID, "an accumulating contraction needs float32 x and a block on the 8-element grid");
  CUtensorMap xmap;
  {
    const size_t xe = xf == X_F16 ? 2 : 4;
    const cuuint64_t xd[3] = {(cuuint64_t)bj, (cuuint64_t)bi, (cuuint64_t)kC};
    const cuuint64_t xs[2] = {(cuuint64_t)ldx * xe, (cuuint64_t)bi * ldx * xe};
    const bool ok = xf == X_F16 ? encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, x, xd, xs, kBoxContractX16,
                                         CU_TENSOR_MAP_SWIZZLE_128B)
                                : encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, x, xd, xs, kBoxContractX,
                                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return fail(c, TM_ERR_CUDA, "tensor map (x, contraction store)");
  }
  p.w = watch(c, KID_CONTRACT, opt);
  cudaError_t e = timed(c, 1, (long long)kC * bi * bj, s,
                        [&] { return launch_contract_bf16(mode, amap, bmap, xmap, p, c->num_sms, s); });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "contraction launch");
}

tm_status run_finish_bf16(tm_ctx* c, const void* x, int ldx, XFormat xf, int x_exp, const float2* zstat, const void* z, int N,
                          int i0, int j0, int bi, int bj, void* out, bool residual, cudaStream_t s,
                          const tm_options* opt) {
  CUtensorMap xmap, zmap;
  {
    const size_t xe = xf == X_F16 ? 2 : 4;
    const cuuint64_t dims[3] = {(cuuint64_t)bj, (cuuint64_t)bi, (cuuint64_t)kC};
    const cuuint64_t str[2] = {(cuuint64_t)ldx * xe, (cuuint64_t)bi * ldx * xe};
    const bool ok = xf == X_F16 ? encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, x, dims, str, kBoxFinishX16,
                                         CU_TENSOR_MAP_SWIZZLE_128B)
                                : encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, x, dims, str, kBoxFinishX,
                                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return fail(c, TM_ERR_CUDA, "tensor map (x)");
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kC, (cuuint64_t)N, (cuuint64_t)N};
    const cuuint64_t str[2] = {(cuuint64_t)kC * 2, (cuuint64_t)N * kC * 2};
    if (!encode(&zmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, z, dims, str, kBoxFinishZ, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (z, finish)");
  }
  // out of this block: base at (i0, j0), extents (128, bj, bi), so that stores clip at the block's edges
  CUtensorMap omap;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kC, (cuuint64_t)bj, (cuuint64_t)bi};
    const cuuint64_t str[2] = {(cuuint64_t)kC * 2, (cuuint64_t)N * kC * 2};
    const void* base = reinterpret_cast<const __nv_bfloat16*>(out) + ((size_t)i0 * N + (size_t)j0) * kC;
    if (!encode(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, kBoxFinishOut, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(c, TM_ERR_CUDA, "tensor map (out, finish)");
  }
  FinishParams p;
  p.x_exp = x_exp;
  p.residual = residual ? 1 : 0;
  p.zstat = zstat;
  std::memcpy(p.cst, c->k3c_host, sizeof p.cst);
  p.inv_scale_o = c->inv_scale_o;
  p.N = N;
  p.i0 = i0;
  p.j0 = j0;
  p.bi = bi;
  p.bj = bj;
  p.tiles_j = (bj + kFinishTileJ - 1) / kFinishTileJ;
  p.total_tiles = (long long)bi * p.tiles_j;
  p.w = watch(c, KID_FINISH, opt);
  cudaError_t e = timed(c, 2, (long long)bi * bj, s,
                        [&] { return launch_finish_bf16(xf == X_F16, xmap, zmap, c->wo_map, c->wg_map, omap, p, c->num_sms, s); });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "finish launch");
}

// Exponent e of the fp16 storage of x. Every x_ij^c = sum_k a b is bounded by N max|a_c| max|b_c|
// <= N ab_bound (the bound from the weights alone, prepare_tensor_core_weights), so with
// e = 14 - ceil(log2(N ab_bound)) every stored value stays below 2^14, four times inside fp16's range:
// the store cannot overflow for any input. e is clamped to [-60, 60] so that 2^(2e) (the LayerNorm
// epsilon in stored units) stays a normal float.
int x16_exponent(const tm_ctx* c, int N) {
  const double bound = (double)N * c->ab_bound;
  if (!(bound > 0)) return 0;
  const int e = 14 - (int)std::ceil(std::log2(bound));
  return std::min(60, std::max(-60, e));
}

tm_status check_common(tm_ctx* c, int N, tm_dtype dtype) {
  if (!c) return TM_ERR_INVALID;
  c->err.clear();
  if (c->layer != 0) return fail(c, TM_ERR_INVALID, "this ctx holds a triangle attention layer (tm_attn_forward)");
  if (N < 1 || N > 65535) return fail(c, TM_ERR_INVALID, "N=%d outside [1, 65535]", N);
  if (dtype != TM_F32 && dtype != TM_BF16) return fail(c, TM_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (dtype == TM_BF16 && !c->tc)
    return fail(c, TM_ERR_UNSUPPORTED, "bf16 needs c_z = c_h = 128 (have %d, %d)", c->c_z, c->c_h);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != c->device) return fail(c, TM_ERR_INVALID, "current device %d is not the ctx's device %d", dev, c->device);
  return check_device_status(c);
}

int choose_block(const tm_ctx* c, int N, const tm_options* opt, size_t ab_bytes, size_t xe) {
  if (opt && opt->block > 0) return std::min(opt->block, N);
  const size_t full_x = (size_t)c->c_h * N * align_up(N, 128 / xe) * xe;
  size_t budget = (size_t)32 << 30;
  const size_t lim = limit_of(c, opt);
  if (lim) budget = lim > ab_bytes ? std::min(budget, lim - ab_bytes) : 0;
  if (full_x <= budget) return N;
  int nb = (N + 2499) / 2500;
  for (;; ++nb) {
    const int B = (int)align_up((size_t)((N + nb - 1) / nb), 8);   // block origins on the 8-element grid
    if ((size_t)c->c_h * B * align_up(B, 128 / xe) * xe <= budget || B <= 256) return B;
  }
}

}  // namespace tmh


// ====================================================================== C ABI

extern "C" {

const char* tm_status_string(tm_status s) {
  const int i = (int)s;
  return (i >= 0 && i < (int)(sizeof kStatusText / sizeof kStatusText[0])) ? kStatusText[i] : "unknown status";
}

const char* tm_last_error(const tm_ctx* ctx) { return ctx ? ctx->err.c_str() : ""; }

long long tm_launch_count(const tm_ctx* ctx) { return ctx ? ctx->launches : 0; }

size_t tm_workspace_bytes(const tm_ctx* ctx) { return ctx ? ctx->ws_bytes : 0; }

tm_status tm_create(int c_z, int c_hidden, const tm_weights* w, tm_ctx** out_ctx) {
  if (!w || !out_ctx) return TM_ERR_INVALID;
  if (c_z < 1 || c_z > 256 || c_hidden < 1 || c_hidden > 256) return TM_ERR_INVALID;
  const float* req[] = {w->ln_in_gamma, w->ln_in_beta, w->w_a, w->w_ga, w->w_b,
                        w->w_gb, w->w_g, w->ln_out_gamma, w->ln_out_beta, w->w_o};
  for (const float* p : req)
    if (!p) return TM_ERR_INVALID;
  tm_ctx* c = new tm_ctx();
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) {
    delete c;
    cudaGetLastError();
    return TM_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  c->c_z = c_z;
  c->c_h = c_hidden;
  if (const char* env = std::getenv("TM_WORKSPACE_LIMIT")) c->env_limit = (size_t)std::strtoull(env, nullptr, 10);

  // float32 weights
  const size_t n_in = c_z, n_h = c_hidden;
  const size_t sizes[10] = {n_in, n_in, n_h * n_in, n_h * n_in, n_h * n_in, n_h * n_in, n_in * n_in, n_h, n_h, n_in * n_h};
  size_t total = 0;
  for (size_t s : sizes) total += align_up(s, 64);
  e = cudaMalloc(&c->w32, total * sizeof(float));
  if (e != cudaSuccess) {
    delete c;
    cudaGetLastError();
    return TM_ERR_CUDA;
  }
  const float* ptrs[10];
  size_t off = 0;
  for (int k = 0; k < 10; ++k) {
    cudaMemcpy(c->w32 + off, req[k], sizes[k] * sizeof(float), cudaMemcpyHostToDevice);
    ptrs[k] = c->w32 + off;
    off += align_up(sizes[k], 64);
  }
  c->f32w = F32Weights{ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[4], ptrs[5], ptrs[6], ptrs[7], ptrs[8], ptrs[9],
                       c_z, c_hidden};

  e = cudaHostAlloc(reinterpret_cast<void**>(&c->status_h), 64, cudaHostAllocMapped);
  if (e != cudaSuccess) {
    tm_destroy(c);
    cudaGetLastError();
    return TM_ERR_CUDA;
  }
  std::memset(c->status_h, 0, 64);
  cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->status_d), c->status_h, 0);

  if (c_z == kC && c_hidden == kC) {
    if (prepare_tensor_core_weights(c, w) != TM_OK) {
      tm_destroy(c);
      return TM_ERR_CUDA;
    }
    c->tc = true;
  }
  *out_ctx = c;
  return TM_OK;
}

void tm_destroy(tm_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  if (c->ws) cudaFree(c->ws);
  if (c->io) cudaFree(c->io);
  if (c->io_in) cudaStreamDestroy(c->io_in);
  if (c->io_out) cudaStreamDestroy(c->io_out);
  for (cudaEvent_t ev : {c->ev_zfree[0], c->ev_zfree[1], c->ev_in, c->ev_out[0], c->ev_out[1]})
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : c->ev_strip) cudaEventDestroy(ev);
  for (void* p : {(void*)c->w32, (void*)c->wk1, (void*)c->k1c, (void*)c->wo16, (void*)c->wg16, c->wbwd, c->ta_w})
    if (p) cudaFree(p);
  if (c->status_h) cudaFreeHost(c->status_h);
  for (auto& t : c->timed) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  for (auto e : c->event_pool) cudaEventDestroy(e);
  cudaGetLastError();
  delete c;
}

tm_status tm_ctx_info(const tm_ctx* c, int* c_z, int* c_hidden, int* layer) {
  if (!c) return TM_ERR_INVALID;
  if (c_z) *c_z = c->c_z;
  if (c_hidden) *c_hidden = c->c_h;
  if (layer) *layer = c->layer;
  return TM_OK;
}

int tm_x_exponent(const tm_ctx* c, int N) {
  if (!c || !c->tc || N < 1) return 0;
  return x16_exponent(c, N);
}

tm_status tm_project_ex(tm_ctx* c, const void* z, const float* mask, int N, tm_dtype dtype, void* a, void* b, int ld,
                        float* zstat, void* stream) {
  tm_status st = check_common(c, N, dtype);
  if (st != TM_OK) return st;
  if (!z || !a || !b || !aligned16(z) || !aligned16(a) || !aligned16(b))
    return fail(c, TM_ERR_INVALID, "z, a, b must be non-null and 16-byte aligned");
  if (mask && (reinterpret_cast<uintptr_t>(mask) & 3u)) return fail(c, TM_ERR_INVALID, "mask must be 4-byte aligned");
  if (ld < N || (dtype == TM_BF16 && ld % 8)) return fail(c, TM_ERR_INVALID, "ld=%d must be >= N (and a multiple of 8 for bf16)", ld);
  if (zstat && dtype != TM_BF16) return fail(c, TM_ERR_INVALID, "zstat is written by the bf16 projection only");
  if (zstat && (reinterpret_cast<uintptr_t>(zstat) & 7u)) return fail(c, TM_ERR_INVALID, "zstat must be 8-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TM_BF16)
    return run_project_bf16(c, z, mask, N, reinterpret_cast<float2*>(zstat), reinterpret_cast<__nv_bfloat16*>(a),
                            reinterpret_cast<__nv_bfloat16*>(b), ld, s, nullptr);
  cudaError_t e = timed(c, 3, (long long)N * N, s, [&] {
    return launch_project_f32(reinterpret_cast<const float*>(z), mask, c->f32w, reinterpret_cast<float*>(a),
                              reinterpret_cast<float*>(b), N, ld, s);
  });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "projection (f32) launch");
}

tm_status tm_project(tm_ctx* c, const void* z, const float* mask, int N, tm_dtype dtype, void* a, void* b, int ld,
                     void* stream) {
  return tm_project_ex(c, z, mask, N, dtype, a, b, ld, nullptr, stream);
}

tm_status tm_contract_ex(tm_ctx* c, const void* a, const void* b, int N, int ld, tm_dtype dtype, tm_direction dir,
                         int i0, int j0, int bi, int bj, void* x, int ldx, int x_storage, void* stream) {
  tm_status st = check_common(c, N, dtype);
  if (st != TM_OK) return st;
  if (dir != TM_OUTGOING && dir != TM_INCOMING) return fail(c, TM_ERR_INVALID, "unknown direction %d", (int)dir);
  if (!a || !b || !x || !aligned16(a) || !aligned16(b) || !aligned16(x))
    return fail(c, TM_ERR_INVALID, "a, b, x must be non-null and 16-byte aligned");
  if (ld < N || (dtype == TM_BF16 && ld % 8)) return fail(c, TM_ERR_INVALID, "bad ld=%d", ld);
  if (i0 < 0 || j0 < 0 || bi < 1 || bj < 1 || i0 + bi > N || j0 + bj > N)
    return fail(c, TM_ERR_INVALID, "block (%d,%d)+(%d,%d) outside the %d x %d grid", i0, j0, bi, bj, N, N);
  if (x_storage != TM_X_FP16 && x_storage != TM_X_FP32) return fail(c, TM_ERR_INVALID, "unknown x_storage %d", x_storage);
  const bool x16 = x_storage == TM_X_FP16;
  if (x16 && dtype != TM_BF16) return fail(c, TM_ERR_INVALID, "fp16 x is a storage of the bf16 path only");
  if (ldx < bj || ldx % (x16 ? 8 : 4))
    return fail(c, TM_ERR_INVALID, "ldx=%d must be >= bj and a multiple of %d", ldx, x16 ? 8 : 4);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool inc = dir == TM_INCOMING;
  if (dtype == TM_BF16)
    return run_contract_bf16(c, a, b, N, ld, inc ? CONTRACT_IN : CONTRACT_OUT, i0, j0, bi, bj, x, ldx, x16 ? X_F16 : X_F32,
                             x16 ? x16_exponent(c, N) : 0, s, nullptr);
  cudaError_t e = timed(c, 3, (long long)c->c_h * bi * bj, s, [&] {
    return launch_contract_f32(inc, reinterpret_cast<const float*>(a), reinterpret_cast<const float*>(b), N, ld,
                               c->c_h, i0, j0, bi, bj, reinterpret_cast<float*>(x), ldx, (long long)bi * ldx, s);
  });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "contraction (f32) launch");
}

tm_status tm_contract(tm_ctx* c, const void* a, const void* b, int N, int ld, tm_dtype dtype, tm_direction dir,
                      int i0, int j0, int bi, int bj, float* x, int ldx, void* stream) {
  return tm_contract_ex(c, a, b, N, ld, dtype, dir, i0, j0, bi, bj, x, ldx, TM_X_FP32, stream);
}

tm_status tm_finish_ex(tm_ctx* c, const void* x, int ldx, int x_storage, const float* zstat, const void* z, int N,
                       tm_dtype dtype, int i0, int j0, int bi, int bj, void* out, void* stream) {
  tm_status st = check_common(c, N, dtype);
  if (st != TM_OK) return st;
  if (!x || !z || !out || !aligned16(x) || !aligned16(z) || !aligned16(out))
    return fail(c, TM_ERR_INVALID, "x, z, out must be non-null and 16-byte aligned");
  if (i0 < 0 || j0 < 0 || bi < 1 || bj < 1 || i0 + bi > N || j0 + bj > N)
    return fail(c, TM_ERR_INVALID, "block outside the grid");
  if (x_storage != TM_X_FP16 && x_storage != TM_X_FP32) return fail(c, TM_ERR_INVALID, "unknown x_storage %d", x_storage);
  const bool x16 = x_storage == TM_X_FP16;
  if (x16 && dtype != TM_BF16) return fail(c, TM_ERR_INVALID, "fp16 x is a storage of the bf16 path only");
  if (x16 && (!zstat || (reinterpret_cast<uintptr_t>(zstat) & 7u)))
    return fail(c, TM_ERR_INVALID, "fp16 x needs the projection's zstat (8-byte aligned)");
  if (ldx < bj || ldx % (x16 ? 8 : 4))
    return fail(c, TM_ERR_INVALID, "ldx=%d must be >= bj and a multiple of %d", ldx, x16 ? 8 : 4);
  const size_t zbytes = (size_t)N * N * c->c_z * (dtype == TM_BF16 ? 2 : 4);
  if (ranges_overlap(z, zbytes, out, zbytes)) return fail(c, TM_ERR_INVALID, "out overlaps z");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TM_BF16)
    return run_finish_bf16(c, x, ldx, x16 ? X_F16 : X_F32, x16 ? x16_exponent(c, N) : 0,
                           reinterpret_cast<const float2*>(zstat), z, N, i0, j0, bi, bj, out, false, s, nullptr);
  cudaError_t e = timed(c, 3, (long long)bi * bj, s, [&] {
    return launch_finish_f32(reinterpret_cast<const float*>(x), ldx, (long long)bi * ldx,
                             reinterpret_cast<const float*>(z), c->f32w, N, i0, j0, bi, bj,
                             reinterpret_cast<float*>(out), false, s);
  });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "finish (f32) launch");
}

tm_status tm_finish(tm_ctx* c, const float* x, int ldx, const void* z, int N, tm_dtype dtype, int i0, int j0, int bi,
                    int bj, void* out, void* stream) {
  return tm_finish_ex(c, x, ldx, TM_X_FP32, nullptr, z, N, dtype, i0, j0, bi, bj, out, stream);
}

tm_status tm_project_block(tm_ctx* c, const void* z, const float* mask_rows, const float* mask_cols, int B, void* a,
                           void* b, int ld, float* zstat, void* stream) {
  tm_status st = check_common(c, B, TM_BF16);
  if (st != TM_OK) return st;
  if (!z || !a || !b || !aligned16(z) || !aligned16(a) || !aligned16(b))
    return fail(c, TM_ERR_INVALID, "z, a, b must be non-null and 16-byte aligned");
  if ((mask_rows && (reinterpret_cast<uintptr_t>(mask_rows) & 3u)) ||
      (mask_cols && (reinterpret_cast<uintptr_t>(mask_cols) & 3u)))
    return fail(c, TM_ERR_INVALID, "masks must be 4-byte aligned");
  if (ld < B || ld % 8) return fail(c, TM_ERR_INVALID, "ld=%d must be >= B and a multiple of 8", ld);
  if (zstat && (reinterpret_cast<uintptr_t>(zstat) & 7u)) return fail(c, TM_ERR_INVALID, "zstat must be 8-byte aligned");
  return run_project_bf16(c, z, mask_rows, B, reinterpret_cast<float2*>(zstat), a, b, ld,
                          reinterpret_cast<cudaStream_t>(stream), nullptr, false, 1.f, 1.f, mask_cols, true);
}

tm_status tm_contract_block(tm_ctx* c, const void* a, const void* b, int B, int ld, tm_direction dir, float* x,
                            int ldx, int accumulate, void* stream) {
  tm_status st = check_common(c, B, TM_BF16);
  if (st != TM_OK) return st;
  if (dir != TM_OUTGOING && dir != TM_INCOMING) return fail(c, TM_ERR_INVALID, "unknown direction %d", (int)dir);
  if (!a || !b || !x || !aligned16(a) || !aligned16(b) || !aligned16(x))
    return fail(c, TM_ERR_INVALID, "a, b, x must be non-null and 16-byte aligned");
  if (ld < B || ld % 8) return fail(c, TM_ERR_INVALID, "ld=%d must be >= B and a multiple of 8", ld);
  if (ldx < B || ldx % 4) return fail(c, TM_ERR_INVALID, "ldx=%d must be >= B and a multiple of 4", ldx);
  if (accumulate != 0 && accumulate != 1) return fail(c, TM_ERR_INVALID, "accumulate must be 0 or 1");
  return run_contract_bf16(c, a, b, B, ld, dir == TM_INCOMING ? CONTRACT_IN : CONTRACT_OUT, 0, 0, B, B, x, ldx, X_F32, 0,
                           reinterpret_cast<cudaStream_t>(stream), nullptr, false, accumulate == 1);
}

tm_status tm_forward_ex(tm_ctx* c, const void* z, const float* mask, int N, tm_dtype dtype, tm_direction dir,
                        void* out, void* stream, const tm_options* opt) {
  tm_status st = check_common(c, N, dtype);
  if (st != TM_OK) return st;
  if (dir != TM_OUTGOING && dir != TM_INCOMING) return fail(c, TM_ERR_INVALID, "unknown direction %d", (int)dir);
  if (!z || !out || !aligned16(z) || !aligned16(out))
    return fail(c, TM_ERR_INVALID, "z and out must be non-null and 16-byte aligned");
  if (mask && (reinterpret_cast<uintptr_t>(mask) & 3u)) return fail(c, TM_ERR_INVALID, "mask must be 4-byte aligned");
  if (opt) {
    for (int r : opt->reserved)
      if (r) return fail(c, TM_ERR_INVALID, "tm_options.reserved must be zero");
    if (opt->block < 0 || opt->timeout_ms < 0) return fail(c, TM_ERR_INVALID, "negative option");
    if (opt->x_storage != TM_X_FP16 && opt->x_storage != TM_X_FP32)
      return fail(c, TM_ERR_INVALID, "unknown x_storage %d", opt->x_storage);
    if (opt->residual != 0 && opt->residual != 1) return fail(c, TM_ERR_INVALID, "residual must be 0 or 1");
  }
  const bool residual = opt && opt->residual;
  // x between the contraction and the finish: scaled fp16 unless float32 is asked for (the float32
  // CUDA-core path always keeps float32)
  const XFormat xf = (dtype == TM_BF16 && !(opt && opt->x_storage == TM_X_FP32)) ? X_F16 : X_F32;
  const size_t esz = dtype == TM_BF16 ? 2 : 4;
  const size_t zbytes = (size_t)N * N * c->c_z * esz;
  const bool in_place = residual && out == z;   // the residual update may overwrite z itself
  if (!in_place && ranges_overlap(z, zbytes, out, zbytes))
    return fail(c, TM_ERR_INVALID, residual ? "out overlaps z without being z" : "out overlaps z");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool inc = dir == TM_INCOMING;

  // Rows of a, b and x start on 128-byte boundaries: a TMA box row then maps onto whole L2 lines
  // (with N = 3605 and 16-byte-aligned rows every 128-byte row segment straddled two lines).
  const int ld = dtype == TM_BF16 ? (int)align_up(N, 64) : N;
  const size_t ab_bytes = align_up((size_t)c->c_h * N * ld * esz, 256);
  const size_t xe = xf == X_F16 ? 2 : 4;
  const int B = choose_block(c, N, opt, 2 * ab_bytes, xe);
  const int ldx = (int)align_up(B, 128 / xe);     // 128-byte rows
  const size_t x_bytes = align_up((size_t)c->c_h * B * ldx * xe, 256);
  // LayerNorm_in statistics per pair, from the projection to the fp16-x finish kernel
  const size_t zst_bytes = xf == X_F16 ? align_up((size_t)N * N * sizeof(float2), 256) : 0;
  st = ensure_workspace(c, 2 * ab_bytes + x_bytes + zst_bytes, s, opt);
  if (st != TM_OK) return st;
  uint8_t* base = reinterpret_cast<uint8_t*>(c->ws);
  void* a = base;
  void* b = base + ab_bytes;
  float* x = reinterpret_cast<float*>(base + 2 * ab_bytes);
  float2* zstat = xf == X_F16 ? reinterpret_cast<float2*>(base + 2 * ab_bytes + x_bytes) : nullptr;

  if (dtype == TM_BF16) {
    const int x_exp = x16_exponent(c, N);
    st = run_project_bf16(c, z, mask, N, zstat, reinterpret_cast<__nv_bfloat16*>(a),
                          reinterpret_cast<__nv_bfloat16*>(b), ld, s, opt);
    if (st != TM_OK) return st;
    if (residual && !in_place) {
      // the finish kernel adds the update to what out holds: give it z first
      cudaError_t e = cudaMemcpyAsync(out, z, zbytes, cudaMemcpyDeviceToDevice, s);
      if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemcpyAsync(out <- z)");
    }
    for (int i0 = 0; i0 < N; i0 += B)
      for (int j0 = 0; j0 < N; j0 += B) {
        const int bi = std::min(B, N - i0), bj = std::min(B, N - j0);
        st = run_contract_bf16(c, reinterpret_cast<const __nv_bfloat16*>(a), reinterpret_cast<const __nv_bfloat16*>(b),
                               N, ld, inc ? CONTRACT_IN : CONTRACT_OUT, i0, j0, bi, bj, x, ldx, xf, x_exp, s, opt);
        if (st != TM_OK) return st;
        st = run_finish_bf16(c, x, ldx, xf, x_exp, zstat, z, N, i0, j0, bi, bj, out, residual, s, opt);
        if (st != TM_OK) return st;
      }
    return TM_OK;
  }
  // float32 CUDA-core path
  cudaError_t e = timed(c, 3, (long long)N * N, s, [&] {
    return launch_project_f32(reinterpret_cast<const float*>(z), mask, c->f32w, reinterpret_cast<float*>(a),
                              reinterpret_cast<float*>(b), N, ld, s);
  });
  if (e != cudaSuccess) return cuda_fail(c, e, "projection (f32) launch");
  for (int i0 = 0; i0 < N; i0 += B)
    for (int j0 = 0; j0 < N; j0 += B) {
      const int bi = std::min(B, N - i0), bj = std::min(B, N - j0);
      e = timed(c, 3, (long long)c->c_h * bi * bj, s, [&] {
        return launch_contract_f32(inc, reinterpret_cast<const float*>(a), reinterpret_cast<const float*>(b), N, ld,
                                   c->c_h, i0, j0, bi, bj, x, ldx, (long long)bi * ldx, s);
      });
      if (e != cudaSuccess) return cuda_fail(c, e, "contraction (f32) launch");
      e = timed(c, 3, (long long)bi * bj, s, [&] {
        return launch_finish_f32(x, ldx, (long long)bi * ldx, reinterpret_cast<const float*>(z), c->f32w, N, i0, j0,
                                 bi, bj, reinterpret_cast<float*>(out), residual, s);
      });
      if (e != cudaSuccess) return cuda_fail(c, e, "finish (f32) launch");
    }
  return TM_OK;
}

tm_status tm_pair_update(tm_ctx* c, void* z, const float* mask, int N, tm_dtype dtype, void* stream,
                         const tm_options* opt) {
  tm_options o{};
  if (opt) o = *opt;
  o.residual = 1;
  tm_status st = tm_forward_ex(c, z, mask, N, dtype, TM_OUTGOING, z, stream, &o);
  if (st != TM_OK) return st;
  return tm_forward_ex(c, z, mask, N, dtype, TM_INCOMING, z, stream, &o);
}

tm_status tm_forward(tm_ctx* c, const void* z, const float* mask, int N, tm_dtype dtype, tm_direction dir, void* out,
                     void* stream) {
  return tm_forward_ex(c, z, mask, N, dtype, dir, out, stream, nullptr);
}

tm_status tm_forward_host(tm_ctx* c, const void* z_host, const float* mask_host, int N, tm_dtype dtype,
                          tm_direction dir, void* out_host, void* stream) {
  tm_status st = check_common(c, N, dtype);
  if (st != TM_OK) return st;
  if (dir != TM_OUTGOING && dir != TM_INCOMING) return fail(c, TM_ERR_INVALID, "unknown direction %d", (int)dir);
  if (!z_host || !out_host) return fail(c, TM_ERR_INVALID, "z_host and out_host must be non-null");
  const size_t esz = dtype == TM_BF16 ? 2 : 4;
  const size_t zbytes = (size_t)N * N * c->c_z * esz;
  if (ranges_overlap(z_host, zbytes, out_host, zbytes)) return fail(c, TM_ERR_INVALID, "out_host overlaps z_host");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // the ctx's copy streams and their events, made on first use
  if (!c->io_in) {
    e = cudaStreamCreateWithFlags(&c->io_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->io_out, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&c->ev_zfree[0], &c->ev_zfree[1], &c->ev_in, &c->ev_out[0], &c->ev_out[1]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(c, e, "copy streams");
  }
  // two staging slots (z, out, mask), used by calls in turn: a call's copy in may then run while the call
  // before it still computes from the other slot
  const size_t zb = align_up(zbytes, 256), mb = align_up((size_t)N * 4, 256);
  const size_t slot_bytes = 2 * zb + mb;
  if (c->io_bytes < 2 * slot_bytes) {
    // nothing of an earlier call may still use the staging buffers when they are replaced
    e = cudaStreamSynchronize(c->io_in);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->io_out);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && c->io) e = cudaFree(c->io);
    if (e != cudaSuccess) return cuda_fail(c, e, "replacing the host-buffer staging");
    c->io = nullptr;
    c->io_bytes = 0;
    e = cudaMalloc(&c->io, 2 * slot_bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      c->io = nullptr;
      return fail(c, TM_ERR_OOM, "cudaMalloc(%zu bytes) for host-buffer staging", 2 * slot_bytes);
    }
    c->io_bytes = 2 * slot_bytes;
  }
  const int slot = c->io_slot;
  uint8_t* zd = reinterpret_cast<uint8_t*>(c->io) + (size_t)slot * slot_bytes;
  uint8_t* od = zd + zb;
  float* md = mask_host ? reinterpret_cast<float*>(zd + 2 * zb) : nullptr;

  // z (and mask) host -> device on io_in, once the kernels of the call that last used this slot are done
  // with it (and, when this z is the last call's output, once that output has landed)
  e = cudaStreamWaitEvent(c->io_in, c->ev_zfree[slot], 0);
  if (e == cudaSuccess && c->last_out_host && ranges_overlap(z_host, zbytes, c->last_out_host, c->last_out_bytes))
    e = cudaStreamWaitEvent(c->io_in, c->ev_out[slot ^ 1], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(zd, z_host, zbytes, cudaMemcpyHostToDevice, c->io_in);
  if (e == cudaSuccess && md) e = cudaMemcpyAsync(md, mask_host, (size_t)N * 4, cudaMemcpyHostToDevice, c->io_in);
  if (e == cudaSuccess) e = cudaEventRecord(c->ev_in, c->io_in);
  // the update on `stream`, after the copy in; what writes this slot's device copy of out also waits for the
  // copy back of the call that last used the slot
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->ev_in, 0);
  if (e != cudaSuccess) return cuda_fail(c, e, "host-to-device copy");

  if (dtype != TM_BF16) {
    if ((e = cudaStreamWaitEvent(s, c->ev_out[slot], 0)) != cudaSuccess) return cuda_fail(c, e, "event");
    st = tm_forward_ex(c, zd, md, N, dtype, dir, od, stream, nullptr);
    if (st != TM_OK) return st;
    e = cudaEventRecord(c->ev_zfree[slot], s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, od, zbytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_out[slot], s);
    if (e != cudaSuccess) return cuda_fail(c, e, "device-to-host copy");
  } else {
    // bf16: the projection over the whole grid, then strips of kStrip rows (contraction, finish), each
    // strip's rows of out copied back on io_out while the next strip computes
    constexpr int kStrip = 512;
    const int ld = (int)align_up(N, 64);
    const int R = std::min(N, kStrip);
    const int ldx = (int)align_up(N, 64);
    const size_t ab_bytes = align_up((size_t)kC * N * ld * 2, 256);
    const size_t x_bytes = align_up((size_t)kC * R * ldx * 2, 256);
    const size_t zst_bytes = align_up((size_t)N * N * sizeof(float2), 256);
    st = ensure_workspace(c, 2 * ab_bytes + x_bytes + zst_bytes, s, nullptr);
    if (st != TM_OK) return st;
    uint8_t* base = reinterpret_cast<uint8_t*>(c->ws);
    void* a = base;
    void* b = base + ab_bytes;
    void* x = base + 2 * ab_bytes;
    float2* zstat = reinterpret_cast<float2*>(base + 2 * ab_bytes + x_bytes);
    const int x_exp = x16_exponent(c, N);
    st = run_project_bf16(c, zd, md, N, zstat, a, b, ld, s, nullptr);
    if (st != TM_OK) return st;
    const int strips = (N + R - 1) / R;
    while ((int)c->ev_strip.size() < strips) {
      cudaEvent_t ev;
      if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(c, e, "event");
      c->ev_strip.push_back(ev);
    }
    const size_t row_bytes = (size_t)N * kC * 2;
    for (int k = 0; k < strips; ++k) {
      const int i0 = k * R, bi = std::min(R, N - i0);
      st = run_contract_bf16(c, a, b, N, ld, dir == TM_INCOMING ? CONTRACT_IN : CONTRACT_OUT, i0, 0, bi, N, x, ldx, X_F16, x_exp, s, nullptr);
      if (st == TM_OK && k == 0 && (e = cudaStreamWaitEvent(s, c->ev_out[slot], 0)) != cudaSuccess)
        return cuda_fail(c, e, "event");
      if (st == TM_OK) st = run_finish_bf16(c, x, ldx, X_F16, x_exp, zstat, zd, N, i0, 0, bi, N, od, false, s, nullptr);
      if (st != TM_OK) return st;
      e = cudaEventRecord(c->ev_strip[k], s);
      if (e == cudaSuccess && k == strips - 1) e = cudaEventRecord(c->ev_zfree[slot], s);   // the last reader of z
      if (e == cudaSuccess) e = cudaStreamWaitEvent(c->io_out, c->ev_strip[k], 0);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(out_host) + (size_t)i0 * row_bytes, od + (size_t)i0 * row_bytes,
                            (size_t)bi * row_bytes, cudaMemcpyDeviceToHost, c->io_out);
      if (e != cudaSuccess) return cuda_fail(c, e, "device-to-host copy");
    }
    e = cudaEventRecord(c->ev_out[slot], c->io_out);
    if (e != cudaSuccess) return cuda_fail(c, e, "event");
  }
  // `stream` waits for the copy back: synchronising it covers out_host
  if ((e = cudaStreamWaitEvent(s, c->ev_out[slot], 0)) != cudaSuccess) return cuda_fail(c, e, "event");
  c->last_out_host = out_host;
  c->last_out_bytes = zbytes;
  c->io_slot = slot ^ 1;
  return TM_OK;
}

tm_status tm_sync_status(tm_ctx* c, void* stream) {
  if (!c) return TM_ERR_INVALID;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamSynchronize");
  return check_device_status(c);
}

tm_status tm_watchdog_selftest(tm_ctx* c, int timeout_ms, void* stream) {
  if (!c) return TM_ERR_INVALID;
  c->err.clear();
  if (timeout_ms < 1 || timeout_ms > 10000) return fail(c, TM_ERR_INVALID, "timeout_ms=%d outside [1, 10000]", timeout_ms);
  tm_options o{};
  o.timeout_ms = timeout_ms;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Watch w = watch(c, KID_SELFTEST, &o);
  cudaError_t e = timed(c, 3, 0, s, [&] { return launch_watchdog_selftest(w, s); });
  return e == cudaSuccess ? TM_OK : cuda_fail(c, e, "self-test launch");
}

tm_status tm_probe_ex2_rate(tm_ctx* c, double* per_second, void* stream) {
  if (!c || !per_second) return TM_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  constexpr int kIters = 20000;
  const int blocks = 4 * c->num_sms;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = launch_probe_ex2(blocks, 1000, s);   // warm-up
  if (e == cudaSuccess) e = cudaEventRecord(e0, s);
  if (e == cudaSuccess) e = launch_probe_ex2(blocks, kIters, s);
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail(c, e, "ex2 probe");
  c->launches += 2;
  *per_second = (double)blocks * 512.0 * 8.0 * kIters / (ms * 1e-3);
  return TM_OK;
}

tm_status tm_set_timing(tm_ctx* c, int enable) {
  if (!c) return TM_ERR_INVALID;
  for (auto& t : c->timed) {
    c->event_pool.push_back(t.start);
    c->event_pool.push_back(t.stop);
  }
  c->timed.clear();
  c->timing = enable != 0;
  return TM_OK;
}

tm_status tm_get_timing(tm_ctx* c, tm_timing* out) {
  if (!c || !out) return TM_ERR_INVALID;
  std::memset(out, 0, sizeof *out);
  for (auto& t : c->timed) {
    cudaError_t e = cudaEventSynchronize(t.stop);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaEventSynchronize");
    float ms = 0.f;
    cudaEventElapsedTime(&ms, t.start, t.stop);
    out->launches[t.kind] += 1;
    out->ms[t.kind] += ms;
    out->units[t.kind] += t.units;
  }
  return TM_OK;
}

}  // extern "C"

// ====================================================================== allocation-free forward
//
// Some callers may not allocate device memory at all: code whose every device
// byte belongs to another allocator (a framework's caching pool, or a fixed
// budget carved out up front), and code that must never pay the host-side stall
// of a device allocation in its steady state. tm_forward_noalloc serves them for
// small grids: the a/b/x scratch of the update lives in one static device array
// of this library (kNoAllocBytes, held by every GPU that loads libtm until the
// process exits), so the call allocates nothing.
namespace {

constexpr int kNoAllocMaxN = 128;
constexpr size_t kNoAllocAB = (size_t)kC * kNoAllocMaxN * kNoAllocMaxN * 2;  // a or b, bf16: 4 MiB
constexpr size_t kNoAllocX = (size_t)kC * kNoAllocMaxN * kNoAllocMaxN * 2;   // x, fp16: 4 MiB
constexpr size_t kNoAllocZst = (size_t)kNoAllocMaxN * kNoAllocMaxN * 8;     // LayerNorm_in statistics: 128 KiB
constexpr size_t kNoAllocBytes = 2 * kNoAllocAB + kNoAllocX + kNoAllocZst;  // 12.125 MiB in all

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch for each device ordinal. The name of the
// array is only a host-side stand-in in host code; the real address is asked
// from the runtime once per device, with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

tm_status noalloc_scratch(tm_ctx* c, uint8_t** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (c->device < 0 || c->device >= kMaxDevices)
    return fail(c, TM_ERR_UNSUPPORTED, "device ordinal %d beyond the no-alloc table", c->device);
  if (!g_noalloc_addr[c->device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(c, e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_addr[c->device] = p;
  }
  *out = reinterpret_cast<uint8_t*>(g_noalloc_addr[c->device]);
  return TM_OK;
}

}  // namespace

extern "C" tm_status tm_forward_noalloc(tm_ctx* c, const void* z, const float* mask, int N, tm_direction dir,
                                        void* out, void* stream) {
  tm_status st = check_common(c, N, TM_BF16);
  if (st != TM_OK) return st;
  if (N > kNoAllocMaxN)
    return fail(c, TM_ERR_UNSUPPORTED, "tm_forward_noalloc handles N <= %d (got N=%d); use tm_forward", kNoAllocMaxN, N);
  if (dir != TM_OUTGOING && dir != TM_INCOMING) return fail(c, TM_ERR_INVALID, "unknown direction %d", (int)dir);
  if (!z || !out || !aligned16(z) || !aligned16(out))
    return fail(c, TM_ERR_INVALID, "z and out must be non-null and 16-byte aligned");
  if (mask && (reinterpret_cast<uintptr_t>(mask) & 3u)) return fail(c, TM_ERR_INVALID, "mask must be 4-byte aligned");
  const size_t zbytes = (size_t)N * N * c->c_z * 2;
  if (ranges_overlap(z, zbytes, out, zbytes)) return fail(c, TM_ERR_INVALID, "out overlaps z");
  uint8_t* scratch = nullptr;
  st = noalloc_scratch(c, &scratch);
  if (st != TM_OK) return st;
  // Every scratch byte the kernels read is written earlier in the same call (a and b
  // for every pair of the grid, x for every entry of the block); the row padding of
  // a/b past N is never read, so nothing has to be cleared between calls. x is kept
  // as tm_forward keeps it by default (fp16, scaled by the same power of two), so
  // that both give the same result.
  const int ld = (int)align_up(N, 8), ldx = (int)align_up(N, 64);
  __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(scratch);
  __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(scratch + kNoAllocAB);
  void* x = scratch + 2 * kNoAllocAB;
  float2* zstat = reinterpret_cast<float2*>(scratch + 2 * kNoAllocAB + kNoAllocX);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool timing = c->timing;  // event creation is an allocation too: no timing inside this call
  c->timing = false;
  const int x_exp = x16_exponent(c, N);
  st = run_project_bf16(c, z, mask, N, zstat, a, b, ld, s, nullptr);
  if (st == TM_OK)
    st = run_contract_bf16(c, a, b, N, ld, dir == TM_INCOMING ? CONTRACT_IN : CONTRACT_OUT, 0, 0, N, N, x, ldx, X_F16, x_exp, s, nullptr);
  if (st == TM_OK) st = run_finish_bf16(c, x, ldx, X_F16, x_exp, zstat, z, N, 0, 0, N, N, out, false, s, nullptr);
  c->timing = timing;
  return st;
}
