// adam_loss.cu -- gs_adam_step, gs_loss_l1 and the small ABI helpers.
//
// Adam (Kingma & Ba, cited in "A Scalable PyTorch Abstraction for Multi-GPU
// Gaussian Splatting", references) with the two moment vectors of the
// per-Gaussian memory figure ("AMD ROCm team open-sources distributed 3D
// Gaussian Splatting training", memory-footprint bullet): one streaming pass
// that reads p, g, m, v and writes p, m, v (28 B per parameter).  HBM-bound;
// 16-byte vector accesses, grid sized to the SM count.
#include <math.h>
#include <stdint.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

struct AdamK {
  float b1, b2, one_m_b1, one_m_b2, step_size, rsqrt_bc2, eps;
};

__device__ __forceinline__ void adam_one(float& p, float g, float& m, float& v, const AdamK& k) {
  m = k.b1 * m + k.one_m_b1 * g;
  v = k.b2 * v + k.one_m_b2 * g * g;
  p -= k.step_size * m / (sqrtf(v) * k.rsqrt_bc2 + k.eps);
}

// With step_dev, the step number (and so the bias corrections) is read from
// device memory; with skip, nothing is updated while the binning status word
// reports an overflow (both for a step captured once and replayed).
__device__ __forceinline__ bool adam_prologue(AdamK& k, const int64_t* step_dev, float lr,
                                              const unsigned int* skip) {
  __shared__ float s_step, s_rbc;
  if (skip && (*reinterpret_cast<const volatile unsigned int*>(skip) & kWsErrCapacity)) return false;
  if (step_dev) {
    if (threadIdx.x == 0) {
      const double t = (double)*step_dev;
      s_step = (float)((double)lr / (1.0 - pow((double)k.b1, t)));
      s_rbc = (float)(1.0 / sqrt(1.0 - pow((double)k.b2, t)));
    }
    __syncthreads();
    k.step_size = s_step;
    k.rsqrt_bc2 = s_rbc;
  }
  return true;
}

__global__ void __launch_bounds__(256) adam_dense_kernel(int64_t count, float* __restrict__ p,
                                                         const float* __restrict__ g,
                                                         float* __restrict__ m,
                                                         float* __restrict__ v, AdamK k,
                                                         const int64_t* __restrict__ step_dev,
                                                         float lr, const unsigned int* skip) {
  if (!adam_prologue(k, step_dev, lr, skip)) return;
  const int64_t n4 = count / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float4* p4 = reinterpret_cast<float4*>(p);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  float4* m4 = reinterpret_cast<float4*>(m);
  float4* v4 = reinterpret_cast<float4*>(v);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 P = p4[i], G = __ldcs(g4 + i), M = m4[i], V = v4[i];
    adam_one(P.x, G.x, M.x, V.x, k);
    adam_one(P.y, G.y, M.y, V.y, k);
    adam_one(P.z, G.z, M.z, V.z, k);
    adam_one(P.w, G.w, M.w, V.w, k);
    p4[i] = P;
    m4[i] = M;
    v4[i] = V;
  }
  for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    adam_one(p[i], g[i], m[i], v[i], k);
}

// Sparse: row-major [59][n], columns with visible == 0 untouched.
__global__ void __launch_bounds__(256) adam_sparse_kernel(int64_t n, float* __restrict__ p,
                                                          const float* __restrict__ g,
                                                          float* __restrict__ m,
                                                          float* __restrict__ v,
                                                          const uint8_t* __restrict__ visible,
                                                          AdamK k,
                                                          const int64_t* __restrict__ step_dev,
                                                          float lr, const unsigned int* skip) {
  if (!adam_prologue(k, step_dev, lr, skip)) return;
  const int64_t row = blockIdx.y;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n; c += stride) {
    if (!visible[c]) continue;
    const int64_t i = row * n + c;
    float P = p[i], M = m[i], V = v[i];
    adam_one(P, g[i], M, V, k);
    p[i] = P;
    m[i] = M;
    v[i] = V;
  }
}

// Sparse, for n a multiple of 4: thread t owns columns 4t..4t+3 of all 59
// rows, reads their visibility once, skips the group when none is visible,
// and otherwise updates the visible lanes of each row with 16-byte accesses
// (the other lanes are written back as read, bit for bit).
__global__ void __launch_bounds__(256) adam_sparse4_kernel(int64_t n, float* __restrict__ p,
                                                           const float* __restrict__ g,
                                                           float* __restrict__ m,
                                                           float* __restrict__ v,
                                                           const uint8_t* __restrict__ visible,
                                                           AdamK k,
                                                           const int64_t* __restrict__ step_dev,
                                                           float lr, const unsigned int* skip) {
  if (!adam_prologue(k, step_dev, lr, skip)) return;
  const int64_t ng = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const uchar4* vis4 = reinterpret_cast<const uchar4*>(visible);
  float4* p4 = reinterpret_cast<float4*>(p);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  float4* m4 = reinterpret_cast<float4*>(m);
  float4* v4 = reinterpret_cast<float4*>(v);
  for (int64_t c4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c4 < ng; c4 += stride) {
    const uchar4 vv = vis4[c4];
    if (!(vv.x | vv.y | vv.z | vv.w)) continue;
#pragma unroll 4
    for (int row = 0; row < GS_NPARAM; ++row) {
      const int64_t i = (int64_t)row * ng + c4;
      float4 P = p4[i], M = m4[i], V = v4[i];
      const float4 G = __ldcs(g4 + i);
      if (vv.x) adam_one(P.x, G.x, M.x, V.x, k);
      if (vv.y) adam_one(P.y, G.y, M.y, V.y, k);
      if (vv.z) adam_one(P.z, G.z, M.z, V.z, k);
      if (vv.w) adam_one(P.w, G.w, M.w, V.w, k);
      p4[i] = P;
      m4[i] = M;
      v4[i] = V;
    }
  }
}

__global__ void __launch_bounds__(256) loss_l1_kernel(int64_t count, const float* __restrict__ img,
                                                      const float* __restrict__ tgt, float inv_count,
                                                      float* __restrict__ loss,
                                                      float* __restrict__ grad) {
  __shared__ float s_w[8];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float acc = 0.f;
  const int64_t n4 = count / 4;
  const float4* a4 = reinterpret_cast<const float4*>(img);
  const float4* b4 = reinterpret_cast<const float4*>(tgt);
  float4* g4 = reinterpret_cast<float4*>(grad);
  auto sgn = [&](float d) { return d > 0.f ? inv_count : (d < 0.f ? -inv_count : 0.f); };
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = __ldcs(a4 + i), b = __ldcs(b4 + i);
    const float4 d = make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
    acc += fabsf(d.x) + fabsf(d.y) + fabsf(d.z) + fabsf(d.w);
    g4[i] = make_float4(sgn(d.x), sgn(d.y), sgn(d.z), sgn(d.w));
  }
  for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const float d = img[i] - tgt[i];
    acc += fabsf(d);
    grad[i] = sgn(d);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < (blockDim.x >> 5) ? s_w[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (threadIdx.x == 0) atomicAdd(loss, w * inv_count);
  }
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 152;
  return sms;
}

}  // namespace
}  // namespace gs

using namespace gs;

static bool adam_args_valid(int64_t step, float beta1, float beta2, float eps) {
  return step >= 1 && beta1 >= 0.f && beta1 < 1.f && beta2 >= 0.f && beta2 < 1.f && eps >= 0.f;
}

// Constants of step `step`, bias corrections in double.
static AdamK make_adam(float lr, float beta1, float beta2, float eps, int64_t step) {
  AdamK k;
  k.b1 = beta1;
  k.b2 = beta2;
  k.one_m_b1 = 1.f - beta1;
  k.one_m_b2 = 1.f - beta2;
  const double bc1 = 1.0 - pow((double)beta1, (double)step);
  const double bc2 = 1.0 - pow((double)beta2, (double)step);
  k.step_size = (float)((double)lr / bc1);
  k.rsqrt_bc2 = (float)(1.0 / sqrt(bc2));
  k.eps = eps;
  return k;
}

static gs_status adam_impl(int64_t n, float* params, const float* grad, float* m, float* v,
                           int64_t step, const int64_t* step_dev, float lr, float beta1,
                           float beta2, float eps, const uint8_t* visible,
                           const unsigned int* skip, void* stream) {
  if (n < 0 || !adam_args_valid(step_dev ? 1 : step, beta1, beta2, eps)) return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  if (!params || !grad || !m || !v || !aligned16(params) || !aligned16(grad) || !aligned16(m) ||
      !aligned16(v))
    return GS_ERR_INVALID_ARG;
  const AdamK k = make_adam(lr, beta1, beta2, eps, step_dev ? 1 : step);
  cudaStream_t st = (cudaStream_t)stream;
  const int sms = sm_count();
  if (!visible) {
    const int64_t count = (int64_t)GS_NPARAM * n;
    const int64_t want = div_up(count / 4 + 1, 256);
    const unsigned blocks = (unsigned)(want < 8 * sms ? want : 8 * sms);
    adam_dense_kernel<<<blocks, 256, 0, st>>>(count, params, grad, m, v, k, step_dev, lr, skip);
  } else if (n % 4 == 0 && (reinterpret_cast<uintptr_t>(visible) & 3u) == 0) {
    const int64_t want = div_up(n / 4, 256);
    const unsigned blocks = (unsigned)(want < 8 * sms ? want : 8 * sms);
    adam_sparse4_kernel<<<blocks, 256, 0, st>>>(n, params, grad, m, v, visible, k, step_dev, lr,
                                                skip);
  } else {
    const int64_t want = div_up(n, 256);
    dim3 grid((unsigned)(want < 2 * sms ? want : 2 * sms), GS_NPARAM);
    adam_sparse_kernel<<<grid, 256, 0, st>>>(n, params, grad, m, v, visible, k, step_dev, lr, skip);
  }
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" gs_status gs_adam_step(int64_t n, float* params, const float* grad, float* m, float* v,
                                  int64_t step, float lr, float beta1, float beta2, float eps,
                                  const uint8_t* visible, void* stream) {
  return adam_impl(n, params, grad, m, v, step, nullptr, lr, beta1, beta2, eps, visible, nullptr,
                   stream);
}

static const unsigned int* status_word(const void* bin_workspace) {
  return bin_workspace ? reinterpret_cast<const unsigned int*>(
                             reinterpret_cast<const unsigned char*>(bin_workspace) + kWsStatusOffset)
                       : nullptr;
}

extern "C" gs_status gs_adam_step_dev(int64_t n, float* params, const float* grad, float* m,
                                      float* v, const int64_t* step, float lr, float beta1,
                                      float beta2, float eps, const uint8_t* visible,
                                      const void* bin_workspace, void* stream) {
  if (!step) return GS_ERR_INVALID_ARG;
  return adam_impl(n, params, grad, m, v, 1, step, lr, beta1, beta2, eps, visible,
                   status_word(bin_workspace), stream);
}

namespace gs {
namespace {
__global__ void step_advance_kernel(int64_t* step, const unsigned int* skip) {
  if (skip && (*reinterpret_cast<const volatile unsigned int*>(skip) & kWsErrCapacity)) return;
  *step += 1;
}
}  // namespace
}  // namespace gs

extern "C" gs_status gs_step_advance(int64_t* step, const void* bin_workspace, void* stream) {
  if (!step) return GS_ERR_INVALID_ARG;
  step_advance_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(step, status_word(bin_workspace));
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" gs_status gs_loss_l1(const float* image, const float* target, int64_t count,
                                float* loss, float* dL_dimage, void* stream) {
  if (count < 0 || !loss) return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  GS_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), st));
  if (count == 0) return GS_OK;
  if (!image || !target || !dL_dimage || !aligned16(image) || !aligned16(target) ||
      !aligned16(dL_dimage))
    return GS_ERR_INVALID_ARG;
  const int sms = sm_count();
  const int64_t want = div_up(count / 4 + 1, 256);
  const unsigned blocks = (unsigned)(want < 4 * sms ? want : 4 * sms);
  loss_l1_kernel<<<blocks, 256, 0, st>>>(count, image, target, (float)(1.0 / (double)count), loss,
                                         dL_dimage);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" const char* gs_status_string(gs_status status) {
  switch (status) {
    case GS_OK: return "ok";
    case GS_ERR_INVALID_ARG: return "invalid argument";
    case GS_ERR_CAPACITY: return "intersection count exceeds capacity";
    case GS_ERR_TIMEOUT: return "a bounded device wait ran out";
    case GS_ERR_CUDA: return "CUDA runtime error";
    case GS_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

extern "C" const char* gs_status_str(gs_status status) { return gs_status_string(status); }

extern "C" int32_t gs_version(void) { return 100; }
