// k_f32.cu -- float32 CUDA-core path of the triangle multiplicative update
// (z, out and every intermediate in float32, FP32 FMA; any 1 <= c_z, c_h <= 256).
//
// Same three steps as the tensor-core path: projection (LayerNorm_in, gated
// masked projections, channel-major a/b), per-channel contraction (shared
// memory tiled), and the output stage (LayerNorm_out, W_o, gate W_g on
// LayerNorm_in(z)). The update is the layer of the code-sample section of
// "NVIDIA BioNeMo escala modelagem biomolecular com context parallelism e
// quebra barreira de memória da GPU".
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int kMaxC = 256;

__device__ __forceinline__ float sigmoid_acc(float v) { return 1.0f / (1.0f + expf(-v)); }

// LayerNorm_in(z_ij) into zh (length c_z), biased variance, eps 1e-5.
__device__ __forceinline__ void layer_norm_in(const float* zp, const F32Weights& w, float* zh) {
  float s = 0.f;
  for (int k = 0; k < w.c_z; ++k) s += zp[k];
  const float mu = s / w.c_z;
  float v = 0.f;
  for (int k = 0; k < w.c_z; ++k) v += (zp[k] - mu) * (zp[k] - mu);
  const float rs = 1.0f / sqrtf(v / w.c_z + 1e-5f);
  for (int k = 0; k < w.c_z; ++k) zh[k] = (zp[k] - mu) * rs * w.ln_in_g[k] + w.ln_in_b[k];
}

__global__ void k1f_project(const float* __restrict__ z, const float* __restrict__ mask, const F32Weights w,
                            float* __restrict__ a, float* __restrict__ b, int N, int ld) {
  const long long pair = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (pair >= (long long)N * N) return;
  const int i = (int)(pair / N), j = (int)(pair - (long long)i * N);
  float zh[kMaxC];
  layer_norm_in(z + pair * w.c_z, w, zh);
  const float m = mask ? mask[i] * mask[j] : 1.0f;
  const size_t chan = (size_t)N * ld;
  for (int h = 0; h < w.c_h; ++h) {
    float pa = 0.f, ga = 0.f, pb = 0.f, gb = 0.f;
    const float *ra = w.w_a + (size_t)h * w.c_z, *rga = w.w_ga + (size_t)h * w.c_z;
    const float *rb = w.w_b + (size_t)h * w.c_z, *rgb = w.w_gb + (size_t)h * w.c_z;
    for (int k = 0; k < w.c_z; ++k) {
      pa = fmaf(ra[k], zh[k], pa);
      ga = fmaf(rga[k], zh[k], ga);
      pb = fmaf(rb[k], zh[k], pb);
      gb = fmaf(rgb[k], zh[k], gb);
    }
    a[h * chan + (size_t)i * ld + j] = sigmoid_acc(ga) * pa * m;
    b[h * chan + (size_t)i * ld + j] = sigmoid_acc(gb) * pb * m;
  }
}

// x[c][i - i0][j - j0] = sum_k A(i, k) B(j, k), with A(i, k) = a[c][i][k], B(j, k) = b[c][j][k]
// (outgoing) or A(i, k) = a[c][k][i], B(j, k) = b[c][k][j] (incoming).
constexpr int T = 16;
__global__ void k2f_contract(const float* __restrict__ a, const float* __restrict__ b, int N, int ld, int i0,
                             int j0, int bi, int bj, float* __restrict__ x, long long ldx, long long chan_stride,
                             int incoming) {
  __shared__ float As[T][T + 1];
  __shared__ float Bs[T][T + 1];
  const int c = blockIdx.z;
  const int ty = threadIdx.y, tx = threadIdx.x;
  const int il = blockIdx.y * T + ty, jl = blockIdx.x * T + tx;
  const size_t chan = (size_t)N * ld;
  const float* ac = a + c * chan;
  const float* bc = b + c * chan;
  float acc = 0.f;
  for (int k0 = 0; k0 < N; k0 += T) {
    // As[r][kk] = A(i0 + blockIdx.y*T + r, k0 + kk); Bs[r][kk] = B(j0 + blockIdx.x*T + r, k0 + kk)
    {
      const int r = ty, kk = tx;
      const int gi = i0 + blockIdx.y * T + r, gk = k0 + kk;
      float va = 0.f;
      if (blockIdx.y * T + r < bi && gk < N) va = incoming ? ac[(size_t)gk * ld + gi] : ac[(size_t)gi * ld + gk];
      As[r][kk] = va;
      const int gj = j0 + blockIdx.x * T + r;
      float vb = 0.f;
      if (blockIdx.x * T + r < bj && gk < N) vb = incoming ? bc[(size_t)gk * ld + gj] : bc[(size_t)gj * ld + gk];
      Bs[r][kk] = vb;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) acc = fmaf(As[ty][kk], Bs[tx][kk], acc);
    __syncthreads();
  }
  if (il < bi && jl < bj) x[c * chan_stride + (long long)il * ldx + jl] = acc;
}

__global__ void k3f_finish(const float* __restrict__ x, long long ldx, long long chan_stride,
                           const float* z, const F32Weights w, int N, int i0, int j0, int bi, int bj,
                           float* out, int residual) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)bi * bj) return;
  const int il = (int)(idx / bj), jl = (int)(idx - (long long)il * bj);
  const int i = i0 + il, j = j0 + jl;
  float xv[kMaxC];
  float s = 0.f;
  for (int c = 0; c < w.c_h; ++c) {
    xv[c] = x[c * chan_stride + (long long)il * ldx + jl];
    s += xv[c];
  }
  const float mu = s / w.c_h;
  float v = 0.f;
  for (int c = 0; c < w.c_h; ++c) v += (xv[c] - mu) * (xv[c] - mu);
  const float rs = 1.0f / sqrtf(v / w.c_h + 1e-5f);
  for (int c = 0; c < w.c_h; ++c) xv[c] = (xv[c] - mu) * rs * w.ln_out_g[c] + w.ln_out_b[c];
  float zh[kMaxC];
  const long long pair = (long long)i * N + j;
  layer_norm_in(z + pair * w.c_z, w, zh);
  float* op = out + pair * w.c_z;
  for (int o = 0; o < w.c_z; ++o) {
    float y = 0.f, g = 0.f;
    const float* ro = w.w_o + (size_t)o * w.c_h;
    const float* rg = w.w_g + (size_t)o * w.c_z;
    for (int c = 0; c < w.c_h; ++c) y = fmaf(ro[c], xv[c], y);
    for (int k = 0; k < w.c_z; ++k) g = fmaf(rg[k], zh[k], g);
    // residual: out = z + update; z of this pair and channel is read before it is written (out may be z)
    // (the product is rounded first, then the sum: the same value as adding z to the plain output)
    const float zo = residual ? z[pair * w.c_z + o] : 0.f;
    op[o] = __fadd_rn(zo, __fmul_rn(sigmoid_acc(g), y));
  }
}

}  // namespace

cudaError_t launch_project_f32(const float* z, const float* mask, const F32Weights& w, float* a, float* b,
                               int N, int ld, cudaStream_t s) {
  const long long pairs = (long long)N * N;
  const int th = 128;
  k1f_project<<<(unsigned)((pairs + th - 1) / th), th, 0, s>>>(z, mask, w, a, b, N, ld);
  return cudaGetLastError();
}

cudaError_t launch_contract_f32(bool incoming, const float* a, const float* b, int N, int ld, int c_h, int i0,
                                int j0, int bi, int bj, float* x, long long ldx, long long chan_stride,
                                cudaStream_t s) {
  dim3 grid((bj + T - 1) / T, (bi + T - 1) / T, c_h), block(T, T);
  k2f_contract<<<grid, block, 0, s>>>(a, b, N, ld, i0, j0, bi, bj, x, ldx, chan_stride, incoming ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_finish_f32(const float* x, long long ldx, long long chan_stride, const float* z,
                              const F32Weights& w, int N, int i0, int j0, int bi, int bj, float* out,
                              bool residual, cudaStream_t s) {
  const long long n = (long long)bi * bj;
  const int th = 128;
  k3f_finish<<<(unsigned)((n + th - 1) / th), th, 0, s>>>(x, ldx, chan_stride, z, w, N, i0, j0, bi, bj, out,
                                                          residual ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace tmk
