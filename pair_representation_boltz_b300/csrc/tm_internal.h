// tm_internal.h -- what the host files of libtm share: the context behind the opaque tm_ctx of the C ABI
// and the helpers that check arguments, encode tensor maps, time launches, hold the workspace and launch
// the update's three bf16 stages. Not part of the public interface (include/tm.h is).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "tm.h"
#include "tm_kernels.h"

namespace tmh {

using namespace tmk;
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn();

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct TimedLaunch {
  cudaEvent_t start, stop;
  int kind;
  long long units;
};

}  // namespace tmh

struct tm_ctx {
  int layer = 0;                 // 0: triangle multiplicative update, 1: triangle attention
  int device = 0, num_sms = 0;
  int c_z = 0, c_h = 0;
  // float32 weights (device), one allocation
  float* w32 = nullptr;
  tmk::F32Weights f32w{};
  // tensor-core path (c_z = c_h = 128)
  bool tc = false;
  __nv_bfloat16* wk1 = nullptr;  // [2 halves][hi, lo][256][128]
  float* k1c = nullptr;          // [2][512]
  __half* wo16 = nullptr;        // [128][128], scaled
  __nv_bfloat16* wg16 = nullptr; // [hi, lo][128][128]
  float k3c_host[4 * tmk::kC] = {};  // finish-kernel constants, passed in its parameter block
  double ab_bound = 0;           // max_c of the bounds on |a_c| and |b_c| multiplied (fp16 x scale)
  float inv_scale_o = 1.f;
  CUtensorMap wk1_map, wo_map, wg_map;
  // backward pass: fp16 images of W_g, W_o, W_a, W_ga, W_b, W_gb (times 2^bwd_wexp[m]) in the
  // 128 x 128 operand-tile layout of the backward kernels, then gamma_in, beta_in, gamma_out, beta_out
  // (float32); bounds on |W_a zh|, |W_b zh| (pv_bound), |zh|, |xh| and |W_o xh| that fix the fp16
  // scales of the backward's operands
  void* wbwd = nullptr;
  int bwd_wexp[6] = {};
  double pv_bound[2] = {}, zh_bound = 0, xh_bound = 0, y_bound = 0;
  // |dL/dx| <= dx_bound * max |dout|: the fp16 scale of the backward's dX
  double dx_bound = 0;
  // triangle attention: fp16 images of W_q, W_k, W_v, W_g, W_o (each scaled by a power of two), then
  // gamma and beta (times the power of two zh is stored with) and W_b (float32); the factors that undo
  // the scales
  void* ta_w = nullptr;
  float ta_wscale[4] = {1.f, 1.f, 1.f, 1.f};
  float ta_oscale = 1.f;
  float ta_bscale = 1.f;
  // status word (mapped host memory)
  int* status_h = nullptr;
  int* status_d = nullptr;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  cudaStream_t ws_stream = nullptr;
  size_t env_limit = 0;
  // device staging of tm_forward_host (two slots, used by calls in turn), its copy streams and events:
  // z in on io_in, out back on io_out (row strips, overlapped with the strips still computing and with
  // the next call's copy in)
  void* io = nullptr;
  size_t io_bytes = 0;
  int io_slot = 0;
  cudaStream_t io_in = nullptr, io_out = nullptr;
  cudaEvent_t ev_zfree[2] = {nullptr, nullptr}, ev_in = nullptr, ev_out[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> ev_strip;
  const void* last_out_host = nullptr;
  size_t last_out_bytes = 0;
  // instrumentation
  bool timing = false;
  std::vector<tmh::TimedLaunch> timed;
  std::vector<cudaEvent_t> event_pool;
  long long launches = 0;
  std::string err;
};

namespace tmh {

tm_status fail(tm_ctx* c, tm_status s, const char* fmt, ...);
tm_status cuda_fail(tm_ctx* c, cudaError_t e, const char* what);
bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const Box& b, CUtensorMapSwizzle sw);
Watch watch(const tm_ctx* c, int kernel, const tm_options* opt);
cudaEvent_t take_event(tm_ctx* c);
tm_status check_device_status(tm_ctx* c);
size_t limit_of(const tm_ctx* c, const tm_options* opt);
tm_status ensure_workspace(tm_ctx* c, size_t bytes, cudaStream_t s, const tm_options* opt);
bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb);
void make_tile_image(const float* W, __nv_bfloat16* img);
void make_tile_image_h(const float* W, double scale, __half* img);
int fp16_image_exponent(const float* W);
// out_f16: a and b leave as fp16 of their bf16 values times scale_a, scale_b (powers of two), for the
// backward pass; ab_f16: the contraction's operands are such fp16 planes.
// mask_col: the token mask of the columns when it differs from the rows' (a block of a grid split into
// blocks); by default the grid's own mask serves both.
tm_status run_project_bf16(tm_ctx* c, const void* z, const float* mask, int N, float2* zstat, void* a,
                           void* b, int ld, cudaStream_t s, const tm_options* opt, bool out_f16 = false,
                           float scale_a = 1.f, float scale_b = 1.f, const float* mask_col = nullptr,
                           bool separate_col_mask = false);
tm_status run_contract_bf16(tm_ctx* c, const void* a, const void* b, int N, int ld, int mode,
                            int i0, int j0, int bi, int bj, void* x, int ldx, XFormat xf, int x_exp,
                            cudaStream_t s, const tm_options* opt, bool ab_f16 = false, bool accumulate = false);
// 2^(target - E) for the exponent E with 2^(E-1) <= bound < 2^E (bound > 0), else 1: the power of two
// that keeps values bounded by `bound` below 2^target.
double pow2_scale_host(double bound, int target);
tm_status run_finish_bf16(tm_ctx* c, const void* x, int ldx, XFormat xf, int x_exp, const float2* zstat, const void* z, int N,
                          int i0, int j0, int bi, int bj, void* out, bool residual, cudaStream_t s,
                          const tm_options* opt);
int x16_exponent(const tm_ctx* c, int N);
tm_status check_common(tm_ctx* c, int N, tm_dtype dtype);
int choose_block(const tm_ctx* c, int N, const tm_options* opt, size_t ab_bytes, size_t xe);

// Launch wrapper: counts launches and, when timing is on, brackets the launch with events on `s`.
template <typename F>
cudaError_t timed(tm_ctx* c, int kind, long long units, cudaStream_t s, F&& launch) {
  TimedLaunch tl{};
  if (c->timing) {
    tl.start = take_event(c);
    tl.stop = take_event(c);
    tl.kind = kind;
    tl.units = units;
    cudaEventRecord(tl.start, s);
  }
  cudaError_t e = launch();
  if (e == cudaSuccess) ++c->launches;
  if (c->timing) {
    cudaEventRecord(tl.stop, s);
    c->timed.push_back(tl);
  }
  return e;
}

}  // namespace tmh
