// k_f32_backward.cu -- float32 CUDA-core backward pass of the triangle multiplicative update
// (every intermediate float32, FP32 FMA; any 1 <= c_z, c_h <= 256).
//
// The gradient is the chain rule through the update's steps in reverse (the layer the
// code-sample section of "NVIDIA BioNeMo escala modelagem biomolecular com context parallelism
// e quebra barreira de memória da GPU" builds, trained at larger crops as its section
// "A pegadinha" asks):
//   output backward (one thread per pair): dy = dout g, dgg = dout y g(1-g), dxh = W_o^T dy,
//     the gate's term W_g^T dgg of dzh, LayerNorm_out backward -> dX (and its transpose);
//   the contraction's gradients come from the float32 contraction kernel with other operands;
//   projection backward (one thread per pair): the gate backward of a and b, the W^T products
//     of dzh and LayerNorm_in backward -> dz;
//   every parameter gradient is a sum over the N^2 pairs of an outer product of two per-pair
//     vectors that the two per-pair kernels store channel-major: outer_sum_f32 forms it
//     in fixed-order partial sums (deterministic, no atomics).
#include "tm_kernels.h"

namespace tmk {
namespace {

constexpr int kMaxC = 256;

__device__ __forceinline__ float sigm(float v) { return 1.0f / (1.0f + expf(-v)); }

// mean and 1/sqrt(var + eps) of v[0..n), biased variance
__device__ __forceinline__ void ln_stats(const float* v, int n, float& mu, float& r) {
  float s = 0.f;
  for (int k = 0; k < n; ++k) s += v[k];
  mu = s / n;
  float q = 0.f;
  for (int k = 0; k < n; ++k) q += (v[k] - mu) * (v[k] - mu);
  r = 1.0f / sqrtf(q / n + 1e-5f);
}

// LayerNorm backward: dv = r (dn - mean(dn) - nrm mean(dn nrm)), dn = dout gamma (in place over d)
__device__ __forceinline__ void ln_backward(float* d, const float* nrm, const float* gamma, float r, int n) {
  float s1 = 0.f, s2 = 0.f;
  for (int k = 0; k < n; ++k) {
    const float dn = d[k] * gamma[k];
    s1 += dn;
    s2 += dn * nrm[k];
  }
  s1 /= n;
  s2 /= n;
  for (int k = 0; k < n; ++k) d[k] = r * (d[k] * gamma[k] - s1 - nrm[k] * s2);
}

__global__ void bo_f32(const float* __restrict__ x, long long ldx, const float* __restrict__ z,
                       const float* __restrict__ dout, const F32Weights w, int N, BwdF32Vectors v) {
  const long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long P = (long long)N * N;
  if (p >= P) return;
  const int i = (int)(p / N), j = (int)(p - (long long)i * N);
  const int Cz = w.c_z, Ch = w.c_h;
  float zh[kMaxC], nx[kMaxC], dy[kMaxC], dgg[kMaxC], dxh[kMaxC];
  {
    const float* zp = z + p * Cz;
    for (int k = 0; k < Cz; ++k) zh[k] = zp[k];
    float mu, r;
    ln_stats(zh, Cz, mu, r);
    for (int k = 0; k < Cz; ++k) zh[k] = (zh[k] - mu) * r * w.ln_in_g[k] + w.ln_in_b[k];
  }
  float rx;
  {
    const long long chan = (long long)N * ldx;
    for (int c = 0; c < Ch; ++c) nx[c] = x[c * chan + (long long)i * ldx + j];
    float mu;
    ln_stats(nx, Ch, mu, rx);
    for (int c = 0; c < Ch; ++c) nx[c] = (nx[c] - mu) * rx;
  }
  for (int o = 0; o < Cz; ++o) {
    float gg = 0.f, y = 0.f;
    const float* rg = w.w_g + (size_t)o * Cz;
    const float* ro = w.w_o + (size_t)o * Ch;
    for (int k = 0; k < Cz; ++k) gg = fmaf(rg[k], zh[k], gg);
    for (int c = 0; c < Ch; ++c) y = fmaf(ro[c], nx[c] * w.ln_out_g[c] + w.ln_out_b[c], y);
    const float g = sigm(gg), d = dout[p * Cz + o];
    dy[o] = d * g;
    dgg[o] = d * y * g * (1.f - g);
  }
  for (int c = 0; c < Ch; ++c) {
    float s = 0.f;
    for (int o = 0; o < Cz; ++o) s = fmaf(w.w_o[(size_t)o * Ch + c], dy[o], s);
    dxh[c] = s;
    v.q_out_n[c * P + p] = s * nx[c];          // d(gamma_out) term
    v.q_out[c * P + p] = s;                    // d(beta_out) term
    v.xh[c * P + p] = nx[c] * w.ln_out_g[c] + w.ln_out_b[c];
  }
  ln_backward(dxh, nx, w.ln_out_g, rx, Ch);
  const long long plane = (long long)N * v.ld;
  for (int c = 0; c < Ch; ++c) {
    v.dX[c * plane + (long long)i * v.ld + j] = dxh[c];
    v.dXT[c * plane + (long long)j * v.ld + i] = dxh[c];
  }
  for (int k = 0; k < Cz; ++k) {
    float s = 0.f;
    for (int o = 0; o < Cz; ++o) s = fmaf(w.w_g[(size_t)o * Cz + k], dgg[o], s);
    v.dzh[k * P + p] = s;
    v.zh[k * P + p] = zh[k];
  }
  for (int o = 0; o < Cz; ++o) {
    v.dy[o * P + p] = dy[o];
    v.dgg[o * P + p] = dgg[o];
  }
}

__global__ void bp_f32(const float* __restrict__ z, const float* __restrict__ mask, const F32Weights w, int N,
                       BwdF32Vectors v, float* __restrict__ dz) {
  const long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long P = (long long)N * N;
  if (p >= P) return;
  const int i = (int)(p / N), k2 = (int)(p - (long long)i * N);
  const int Cz = w.c_z, Ch = w.c_h;
  float nz[kMaxC], zh[kMaxC], dzh[kMaxC];
  float rz;
  {
    const float* zp = z + p * Cz;
    for (int k = 0; k < Cz; ++k) nz[k] = zp[k];
    float mu;
    ln_stats(nz, Cz, mu, rz);
    for (int k = 0; k < Cz; ++k) {
      nz[k] = (nz[k] - mu) * rz;
      zh[k] = nz[k] * w.ln_in_g[k] + w.ln_in_b[k];
      dzh[k] = v.dzh[k * P + p];
    }
  }
  const float m = mask ? mask[i] * mask[k2] : 1.0f;
  const long long plane = (long long)N * v.ld;
  for (int h = 0; h < Ch; ++h) {
    const float *ra = w.w_a + (size_t)h * Cz, *rga = w.w_ga + (size_t)h * Cz;
    const float *rb = w.w_b + (size_t)h * Cz, *rgb = w.w_gb + (size_t)h * Cz;
    float pa = 0.f, ga = 0.f, pb = 0.f, gb = 0.f;
    for (int k = 0; k < Cz; ++k) {
      pa = fmaf(ra[k], zh[k], pa);
      ga = fmaf(rga[k], zh[k], ga);
      pb = fmaf(rb[k], zh[k], pb);
      gb = fmaf(rgb[k], zh[k], gb);
    }
    const float sa = sigm(ga), sb = sigm(gb);
    const float da = v.dA[h * plane + (long long)i * v.ld + k2] * m;
    const float db = v.dB[h * plane + (long long)i * v.ld + k2] * m;
    const float dpa = da * sa, dga = da * pa * sa * (1.f - sa);
    const float dpb = db * sb, dgb = db * pb * sb * (1.f - sb);
    v.dpa[h * P + p] = dpa;
    v.dga[h * P + p] = dga;
    v.dpb[h * P + p] = dpb;
    v.dgb[h * P + p] = dgb;
    for (int k = 0; k < Cz; ++k)
      dzh[k] += ra[k] * dpa + rga[k] * dga + rb[k] * dpb + rgb[k] * dgb;
  }
  for (int k = 0; k < Cz; ++k) {
    v.q_in_n[k * P + p] = dzh[k] * nz[k];      // d(gamma_in) term
    v.q_in[k * P + p] = dzh[k];                // d(beta_in) term
  }
  ln_backward(dzh, nz, w.ln_in_g, rz, Cz);
  for (int k = 0; k < Cz; ++k) dz[p * Cz + k] = dzh[k];
}

// part[s][o][k] = sum over p in split s of U[o][p] V[k][p] (V == nullptr: V = 1, K = 1)
constexpr int OT = 16;
__global__ void outer_sum_f32(const float* __restrict__ U, const float* __restrict__ V, int O, int K, long long P,
                              long long chunk, float* __restrict__ part) {
  __shared__ float Us[OT][OT + 1];
  __shared__ float Vs[OT][OT + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int o = blockIdx.y * OT + ty, k = blockIdx.x * OT + tx;
  const long long p0 = (long long)blockIdx.z * chunk;
  const long long p1 = p0 + chunk < P ? p0 + chunk : P;
  float acc = 0.f;
  for (long long q = p0; q < p1; q += OT) {
    // Us[r][t] = U[blockIdx.y*OT + r][q + t]; Vs[r][t] = V[blockIdx.x*OT + r][q + t]
    {
      const int r = ty, t = tx;
      const long long pp = q + t;
      const int uo = blockIdx.y * OT + r, vk = blockIdx.x * OT + r;
      Us[r][t] = (uo < O && pp < p1) ? U[(long long)uo * P + pp] : 0.f;
      Vs[r][t] = (vk < K && pp < p1) ? (V ? V[(long long)vk * P + pp] : 1.f) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < OT; ++t) acc = fmaf(Us[ty][t], Vs[tx][t], acc);
    __syncthreads();
  }
  if (o < O && k < K) part[((long long)blockIdx.z * O + o) * K + k] = acc;
}

__global__ void sum_parts_f32(const float* __restrict__ part, int S, long long E, long long stride,
                              float* __restrict__ out) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  float s = 0.f;
  for (int q = 0; q < S; ++q) s += part[q * stride + e];
  out[e] = s;
}

}  // namespace

cudaError_t launch_bwd_output_f32(const float* x, long long ldx, const float* z, const float* dout,
                                  const F32Weights& w, int N, const BwdF32Vectors& v, cudaStream_t s) {
  const long long P = (long long)N * N;
  const int th = 128;
  bo_f32<<<(unsigned)((P + th - 1) / th), th, 0, s>>>(x, ldx, z, dout, w, N, v);
  return cudaGetLastError();
}

cudaError_t launch_bwd_project_f32(const float* z, const float* mask, const F32Weights& w, int N,
                                   const BwdF32Vectors& v, float* dz, cudaStream_t s) {
  const long long P = (long long)N * N;
  const int th = 128;
  bp_f32<<<(unsigned)((P + th - 1) / th), th, 0, s>>>(z, mask, w, N, v, dz);
  return cudaGetLastError();
}

int outer_sum_splits(long long P) {
  long long S = (P + 16383) / 16384;
  return (int)(S < 1 ? 1 : (S > kOuterSumMaxSplits ? kOuterSumMaxSplits : S));
}

cudaError_t launch_outer_sum_f32(const float* U, const float* V, int O, int K, long long P, float* part,
                                 float* out, cudaStream_t s) {
  const int S = outer_sum_splits(P);
  const long long chunk = (P + S - 1) / S;
  dim3 grid((K + OT - 1) / OT, (O + OT - 1) / OT, S), block(OT, OT);
  outer_sum_f32<<<grid, block, 0, s>>>(U, V, O, K, P, chunk, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_sum_parts(part, S, (long long)O * K, (long long)O * K, out, s);
}

namespace {
// One launch for several partial-sum jobs (blockIdx.y = job); the loads of a thread are independent,
// the sum runs over q = 0, 1, ... in order.
__global__ void sum_parts_multi(const SumJobs j, int S) {
  const int k = blockIdx.y;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= j.E[k] || !j.out[k]) return;
  const float* src = j.part[k] + e;
  const long long st = j.stride[k];
  float s = 0.f;
#pragma unroll 8
  for (int q = 0; q < S; ++q) s += src[q * st];
  j.out[k][e] = s;
}
}  // namespace

cudaError_t launch_sum_parts_multi(const SumJobs& j, int S, cudaStream_t s) {
  long long emax = 0;
  for (int k = 0; k < j.n; ++k) emax = j.E[k] > emax ? j.E[k] : emax;
  if (j.n == 0 || emax == 0) return cudaSuccess;
  dim3 grid((unsigned)((emax + 127) / 128), (unsigned)j.n);
  sum_parts_multi<<<grid, 128, 0, s>>>(j, S);
  return cudaGetLastError();
}

cudaError_t launch_sum_parts(const float* part, int S, long long E, long long stride, float* out, cudaStream_t s) {
  sum_parts_f32<<<(unsigned)((E + 255) / 256), 256, 0, s>>>(part, S, E, stride, out);
  return cudaGetLastError();
}

}  // namespace tmk
