// pa_merge.cu -- pa_lse_merge: the log-sum-exp merge of attention partials, the combine
// step of a context split across GPUs.  See include/pa.h for the contract.
//
// HBM-bound: each (row, head) vector reads its num_parts partial outputs (fp32, 512 B each)
// and lse words once and writes one output.  One warp per vector, four head_dim values
// (one float4) per lane; the lse words are read by every lane of the warp (a broadcast).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"

namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;  // vectors per CTA
constexpr int kMaxParts = 64;

struct MergeParams {
  const float4 *part_out;
  const float *part_lse;
  void *out;
  float *lse;
  int64_t num_vecs;  // rows * heads
  int32_t num_parts, out_f32;
};

__global__ void __launch_bounds__(kWarps * 32) lse_merge_kernel(const MergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t v = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (v >= p.num_vecs) return;
  float M = -INFINITY;
  for (int i = 0; i < p.num_parts; ++i) M = fmaxf(M, __ldg(p.part_lse + (int64_t)i * p.num_vecs + v));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (M != -INFINITY) {
    const int64_t stride = p.num_vecs * (kD / 4);  // float4s per part
    const float4 *src = p.part_out + v * (kD / 4) + lane;
    int i = 0;
    for (; i + 4 <= p.num_parts; i += 4) {  // four parts' loads in flight together
      float w[4];
      float4 x[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float l = __ldg(p.part_lse + (int64_t)(i + k) * p.num_vecs + v);
        w[k] = l == -INFINITY ? 0.f : __expf(l - M);
        x[k] = __ldg(src + (int64_t)(i + k) * stride);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        z += w[k];
        if (w[k] != 0.f) {  // an empty part's output may be anything: it does not enter
          acc.x = fmaf(w[k], x[k].x, acc.x);
          acc.y = fmaf(w[k], x[k].y, acc.y);
          acc.z = fmaf(w[k], x[k].z, acc.z);
          acc.w = fmaf(w[k], x[k].w, acc.w);
        }
      }
    }
    for (; i < p.num_parts; ++i) {
      const float l = __ldg(p.part_lse + (int64_t)i * p.num_vecs + v);
      if (l == -INFINITY) continue;
      const float w = __expf(l - M);
      const float4 x = __ldg(src + (int64_t)i * stride);
      z += w;
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
    const float s = 1.f / z;
    acc.x *= s;
    acc.y *= s;
    acc.z *= s;
    acc.w *= s;
  }
  if (p.out_f32) {
    reinterpret_cast<float4 *>(p.out)[v * (kD / 4) + lane] = acc;
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t *>(&a);
    w.y = *reinterpret_cast<const uint32_t *>(&b);
    reinterpret_cast<uint2 *>(p.out)[v * (kD / 4) + lane] = w;
  }
  if (p.lse != nullptr && lane == 0) p.lse[v] = M == -INFINITY ? -INFINITY : M + __logf(z);
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

}  // namespace

extern "C" pa_status_t pa_lse_merge(const pa_lse_merge_args_t *a, void *stream) {
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  if (a->reserved != 0 || a->num_rows < 0 || a->num_heads < 1 || a->num_parts < 1)
    return PA_ERR_INVALID_ARG;
  if (a->num_parts > kMaxParts || a->head_dim != kD) return PA_ERR_UNSUPPORTED;
  if (a->out_dtype != PA_OUT_BF16 && a->out_dtype != PA_OUT_F32) return PA_ERR_INVALID_ARG;
  if (a->num_rows == 0) return PA_OK;
  if (a->part_out == nullptr || a->part_lse == nullptr || a->out == nullptr)
    return PA_ERR_INVALID_ARG;
  if (!aligned(a->part_out, 16) || !aligned(a->out, 16) || !aligned(a->part_lse, 4) ||
      (a->lse != nullptr && !aligned(a->lse, 4)))
    return PA_ERR_ALIGN;
  MergeParams p;
  p.part_out = reinterpret_cast<const float4 *>(a->part_out);
  p.part_lse = a->part_lse;
  p.out = a->out;
  p.lse = a->lse;
  p.num_vecs = (int64_t)a->num_rows * a->num_heads;
  p.num_parts = a->num_parts;
  p.out_f32 = a->out_dtype == PA_OUT_F32;
  const int64_t blocks = (p.num_vecs + kWarps - 1) / kWarps;
  if (blocks > INT32_MAX) return PA_ERR_INVALID_ARG;
  (void)cudaGetLastError();  // drop an earlier, unrelated launch error
  lse_merge_kernel<<<(unsigned)blocks, kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
