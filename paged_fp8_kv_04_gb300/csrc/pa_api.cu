// pa_api.cu -- host side of libpagedfp8: plan sizing and validation, the launch of the
// decode kernel, and the test hooks.  See include/pa.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>

#include "pa.h"
#include "pa_decode_kernel.cuh"
#include "pa_umma.cuh"

namespace {

constexpr int kMaxBatch = 4096;
constexpr int kMaxSmemDefault = 232448;  // 227 KB opt-in per CTA on sm_100-class parts
constexpr double kLog2e = 1.4426950408889634;
constexpr int kSmallXSlots = 2;  // exchange slots of plans with at most two query tokens

struct Geometry {
  int num_sms = 0, grid = 0, nstage = 0, ppt = 0, ps_shift = 0, mmax = 0;
  int maxch = 0, part_tiles = 0, max_tiles = 0, stage_bytes = 0, qslot_bytes = 0;
  int off_q = 0, off_merge = 0, off_tstart = 0, off_meta = 0, off_bar = 0, off_misc = 0;
  int xslots = 4;
  int64_t slots = 0;
  size_t smem = 0, ws = 0, off_status = 0, off_counters = 0, off_flags = 0, off_ml = 0, off_o = 0;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

pa_status_t validate(const pa_plan_desc_t *d) {
  if (d == nullptr) return PA_ERR_INVALID_ARG;
  for (int k = 0; k < 2; ++k)
    if (d->reserved[k] != 0) return PA_ERR_INVALID_ARG;
  if ((d->flags & ~(PA_PLAN_NO_PDL | PA_PLAN_TCGEN05)) != 0) return PA_ERR_INVALID_ARG;
  if (d->num_kv_heads < 1 || d->num_kv_heads > 64) return PA_ERR_UNSUPPORTED;
  if (d->group_size != pa::kG) return PA_ERR_UNSUPPORTED;
  if (d->head_dim != pa::kD) return PA_ERR_UNSUPPORTED;
  if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64 && d->page_size != 128)
    return PA_ERR_UNSUPPORTED;
  if (d->kv_dtype == PA_KV_FP8_E4M3) {
    if (d->scale_mode != PA_SCALE_SCALAR && d->scale_mode != PA_SCALE_PER_TOKEN)
      return PA_ERR_UNSUPPORTED;
  } else if (d->kv_dtype == PA_KV_BF16) {
    if (d->scale_mode != PA_SCALE_NONE) return PA_ERR_UNSUPPORTED;
  } else {
    return PA_ERR_INVALID_ARG;
  }
  if (d->q_mode != PA_Q_UNIFORM && d->q_mode != PA_Q_RAGGED) return PA_ERR_INVALID_ARG;
  if (d->q_len < 1) return PA_ERR_INVALID_ARG;
  if (d->q_len > pa::kMaxQ) return PA_ERR_UNSUPPORTED;
  if (d->max_batch < 1) return PA_ERR_INVALID_ARG;
  if (d->max_batch > kMaxBatch) return PA_ERR_UNSUPPORTED;
  if (d->max_rows < 1) return PA_ERR_INVALID_ARG;
  if (d->max_context_len < 1) return PA_ERR_INVALID_ARG;
  if (d->max_selected_pages < 0) return PA_ERR_INVALID_ARG;
  if (d->partition_tokens < 0) return PA_ERR_INVALID_ARG;
  if (d->partition_tokens > 0 && d->partition_tokens % pa::kTile != 0) return PA_ERR_UNSUPPORTED;
  if (d->out_dtype != PA_OUT_BF16 && d->out_dtype != PA_OUT_F32) return PA_ERR_INVALID_ARG;
  if (d->num_sms < 0) return PA_ERR_INVALID_ARG;
  // Tile and position counts are held in int32 on the device.
  const int64_t pages = (d->max_context_len + (int64_t)d->page_size - 1) / d->page_size;
  if (pages * d->page_size > INT32_MAX / 2) return PA_ERR_UNSUPPORTED;
  const int64_t tiles = std::max<int64_t>((d->max_context_len + pa::kTile - 1) / pa::kTile,
                                          (d->max_selected_pages + 128 / d->page_size - 1) /
                                              (128 / d->page_size));
  if (tiles * d->max_batch * d->num_kv_heads > INT32_MAX / 2) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

pa_status_t device_sms(int *sms, int *smem_optin) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaDeviceGetAttribute(smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

bool use_umma(const pa_plan_desc_t &d);

pa_status_t geometry(const pa_plan_desc_t *d, Geometry *g) {
  pa_status_t st = validate(d);
  if (st != PA_OK) return st;
  int sms = d->num_sms, smem_max = kMaxSmemDefault;
  if (sms == 0) {
    st = device_sms(&sms, &smem_max);
    if (st != PA_OK) return st;
  }
  g->num_sms = sms;
  g->ppt = pa::kTile / d->page_size;
  g->ps_shift = log2i(d->page_size);
  g->mmax = pa::kG * d->q_len;
  g->max_tiles = (int)std::max<int64_t>((d->max_context_len + pa::kTile - 1) / pa::kTile,
                                        (d->max_selected_pages + g->ppt - 1) / g->ppt);
  if (d->partition_tokens == 0) {
    g->grid = sms;
    g->maxch = 1;
    g->part_tiles = 0;
  } else {
    g->part_tiles = d->partition_tokens / pa::kTile;
    g->maxch = (g->max_tiles + g->part_tiles - 1) / g->part_tiles;
    const int64_t grid = (int64_t)d->max_batch * d->num_kv_heads * g->maxch;
    if (grid > (1 << 22)) return PA_ERR_UNSUPPORTED;
    g->grid = (int)grid;
  }
  g->slots = 2 * (int64_t)g->grid;

  // Shared memory: stages | 2 query slots | merge buffer | tile prefix | meta | barriers | misc
  g->stage_bytes = d->kv_dtype == PA_KV_FP8_E4M3 ? (2 * pa::kTile * pa::kD + 1024)
                                                 : (4 * pa::kTile * pa::kD);
  g->qslot_bytes = d->q_len * pa::kQRowBytes;
  // The exchange buffer (mid-stream ends; the CTA's last merge runs in stage memory) has 4
  // slots, or 2 for plans of at most two query tokens on the mma.sync kernel (a round moves
  // whole slices, q_len m-tiles each) where that leaves room for one more stage: two slots
  // take more rounds per mid-stream end.
  auto fit = [&](int xslots, bool commit) {
    const size_t merge_bytes = (size_t)xslots * (8192 + 512);
    for (int ns = 6; ns >= 2; --ns) {
      size_t off = (size_t)ns * g->stage_bytes;
      const size_t off_q = off;
      off += 2 * (size_t)g->qslot_bytes;
      const size_t off_merge = off;
      off += merge_bytes;
      const size_t off_tstart = off;
      off += round_up((size_t)(2 * d->max_batch + 4) * 4, 16);  // tstart, then the CTA prefix
      const size_t off_meta = off;
      off += (size_t)ns * sizeof(pa::StageMeta);
      const size_t off_bar = off;
      off += round_up((size_t)(2 * ns + 3 + pa::kUmmaBars) * 8, 16);
      const size_t off_misc = off;
      off += pa::kMiscBytes;
      const size_t total = off + 1024;  // slack for the 1024-byte alignment of the base
      if (total <= (size_t)smem_max) {
        if (commit) {
          g->xslots = xslots;
          g->nstage = ns;
          g->off_q = (int)off_q;
          g->off_merge = (int)off_merge;
          g->off_tstart = (int)off_tstart;
          g->off_meta = (int)off_meta;
          g->off_bar = (int)off_bar;
          g->off_misc = (int)off_misc;
          g->smem = total;
        }
        return ns;
      }
    }
    return 0;
  };
  const bool small = d->q_len <= 2 && !use_umma(*d);
  fit(small && fit(kSmallXSlots, false) > fit(4, false) ? kSmallXSlots : 4, true);
  if (g->nstage == 0) return PA_ERR_UNSUPPORTED;

  size_t off = 0;
  g->off_status = off;
  off += 256;
  g->off_counters = off;
  off = round_up(off + (size_t)d->max_batch * d->num_kv_heads * 4, 256);
  g->off_flags = off;
  off = round_up(off + (size_t)d->max_batch * d->num_kv_heads * 4, 256);
  g->off_ml = off;
  off = round_up(off + (size_t)g->slots * 2 * g->mmax * 4, 256);
  g->off_o = off;
  off = round_up(off + (size_t)g->slots * g->mmax * pa::kD * 4, 256);
  g->ws = off;
  return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D map over a cache viewed as [num_pages * Hkv * page_size rows][head_dim elements],
// box = one page of rows, 128-byte swizzle (a BF16 row is loaded as two 64-element boxes).
bool encode_cache_map(CUtensorMap *m, const void *ptr, int64_t rows, int kv_dtype, int ps) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
  cuuint64_t dims[2] = {(cuuint64_t)pa::kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(fp8 ? pa::kD : 2 * pa::kD)};
  cuuint32_t box[2] = {(cuuint32_t)(fp8 ? 128 : 64), (cuuint32_t)ps};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

struct pa_plan {
  pa_plan_desc_t desc;
  Geometry geo;
  int device = 0;
  void *ws = nullptr;
  std::mutex mu;
  const void *tk = nullptr, *tv = nullptr;
  int64_t tpages = -1;
  CUtensorMap tmk, tmv;
};

namespace {

// Also checks the build's register count: the kernel's register split assumes the
// launch allocation of exactly kLaunchRegs per thread (any other count is refused).
template <int KVT, int SM, bool DUMP>
cudaError_t set_smem_attr(size_t smem) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, pa::decode_kernel<KVT, SM, DUMP>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != pa::kLaunchRegs) return cudaErrorInvalidKernelImage;
  return cudaFuncSetAttribute(pa::decode_kernel<KVT, SM, DUMP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// The tcgen05 kernel serves FP8 plans whose requests have one query token, on request.
bool use_umma(const pa_plan_desc_t &d) {
  return d.kv_dtype == PA_KV_FP8_E4M3 && d.q_len == 1 && (d.flags & PA_PLAN_TCGEN05) != 0;
}

template <int SM>
cudaError_t set_umma_attr(size_t smem) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, pa::decode_umma_kernel<SM>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != pa::kLaunchRegs) return cudaErrorInvalidKernelImage;
  return cudaFuncSetAttribute(pa::decode_umma_kernel<SM>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t prepare_kernels(const pa_plan_desc_t &d, size_t smem) {
  cudaError_t e;
  if (use_umma(d)) {
    e = d.scale_mode == PA_SCALE_SCALAR ? set_umma_attr<PA_SCALE_SCALAR>(smem)
                                        : set_umma_attr<PA_SCALE_PER_TOKEN>(smem);
    if (e != cudaSuccess) return e;
  }
  if (d.kv_dtype == PA_KV_BF16) {
    if ((e = set_smem_attr<PA_KV_BF16, PA_SCALE_NONE, false>(smem)) != cudaSuccess) return e;
    return set_smem_attr<PA_KV_BF16, PA_SCALE_NONE, true>(smem);
  }
  if (d.scale_mode == PA_SCALE_SCALAR) {
    if ((e = set_smem_attr<PA_KV_FP8_E4M3, PA_SCALE_SCALAR, false>(smem)) != cudaSuccess) return e;
    return set_smem_attr<PA_KV_FP8_E4M3, PA_SCALE_SCALAR, true>(smem);
  }
  if ((e = set_smem_attr<PA_KV_FP8_E4M3, PA_SCALE_PER_TOKEN, false>(smem)) != cudaSuccess) return e;
  return set_smem_attr<PA_KV_FP8_E4M3, PA_SCALE_PER_TOKEN, true>(smem);
}

// Fills every kernel parameter except the tensor maps and the dump.
void fill_params(const pa_plan *plan, const pa_decode_args_t *a, pa::KParams *k) {
  const pa_plan_desc_t &d = plan->desc;
  const Geometry &g = plan->geo;
  uint8_t *ws = static_cast<uint8_t *>(plan->ws);
  k->q = static_cast<const uint16_t *>(a->q);
  k->k_cache = static_cast<const uint8_t *>(a->k_cache);
  k->v_cache = static_cast<const uint8_t *>(a->v_cache);
  k->k_scale = a->k_scale;
  k->v_scale = a->v_scale;
  k->block_table = a->block_table;
  k->context_lens = a->context_lens;
  k->cu_q = a->cu_seqlens_q;
  k->sel = a->selected_pages;
  k->nsel = a->num_selected;
  k->out = a->out;
  k->lse = a->lse;
  k->status = reinterpret_cast<uint32_t *>(ws + g.off_status);
  k->counters = reinterpret_cast<int32_t *>(ws + g.off_counters);
  k->flags = reinterpret_cast<int32_t *>(ws + g.off_flags);
  k->part_ml = reinterpret_cast<float *>(ws + g.off_ml);
  k->part_o = reinterpret_cast<float *>(ws + g.off_o);
  k->dump = nullptr;
  k->dump_tiles = 0;
  k->num_pages = a->num_pages;
  const double sl2 = (double)a->sm_scale * kLog2e;
  if (d.kv_dtype == PA_KV_BF16) {
    k->kfold = (float)sl2;
    k->pfold = 1.f;
    k->vpost = 1.f;
  } else if (d.scale_mode == PA_SCALE_SCALAR) {
    // Scalar scales: K's folds into the score scale, V's multiplies the normalised
    // output once (vLLM PR 52060, "Suggested Fix").
    k->kfold = (float)((double)a->k_scale_scalar * sl2);
    k->pfold = 1.f;
    k->vpost = a->v_scale_scalar * (1.f / 256.f);  // P' of the mma.sync kernel carries 2^8
  } else {
    // Per-token scales: k_scale[token] multiplies the score column, v_scale[token] the
    // P column, relative to a power of two that the kernel keeps per warp and undoes
    // before the output.
    k->kfold = (float)sl2;
    k->pfold = 1.f;
    k->vpost = 1.f;
  }
  k->num_seqs = a->num_seqs;
  k->Hkv = d.num_kv_heads;
  k->ps = d.page_size;
  k->ps_shift = g.ps_shift;
  k->ppt = g.ppt;
  k->bt_stride = a->block_table_stride;
  k->sel_stride = a->selected_pages ? a->selected_stride : 0;
  k->q_uniform = d.q_mode == PA_Q_UNIFORM ? d.q_len : 0;
  k->max_q = d.q_len;
  k->max_ctx = d.max_context_len;
  k->num_rows = a->num_rows;
  k->out_f32 = d.out_dtype == PA_OUT_F32;
  k->sched_partition = d.partition_tokens > 0;
  k->part_tiles = g.part_tiles;
  k->maxch = g.maxch;
  k->grid = d.partition_tokens > 0 ? a->num_seqs * d.num_kv_heads * g.maxch : g.grid;
  // one CTA per SM (the launch bound and the shared-memory carve allow no more), so a grid
  // no larger than the SM count is resident at once
  k->coresident = k->grid <= g.num_sms ? 1 : 0;
  k->nstage = g.nstage;
  k->mmax = g.mmax;
  k->sparse = a->selected_pages != nullptr;
  k->off_q = g.off_q;
  k->qslot_bytes = g.qslot_bytes;
  k->off_merge = g.off_merge;
  k->off_tstart = g.off_tstart;
  k->off_meta = g.off_meta;
  k->off_bar = g.off_bar;
  k->off_misc = g.off_misc;
  k->stage_bytes = g.stage_bytes;
  k->xslots = g.xslots;
}

pa_status_t tensor_maps(pa_plan *plan, const pa_decode_args_t *a, pa::KParams *k) {
  std::lock_guard<std::mutex> lk(plan->mu);
  if (plan->tk != a->k_cache || plan->tv != a->v_cache || plan->tpages != a->num_pages) {
    const int64_t rows = a->num_pages * plan->desc.num_kv_heads * plan->desc.page_size;
    if (!encode_cache_map(&plan->tmk, a->k_cache, rows, plan->desc.kv_dtype, plan->desc.page_size) ||
        !encode_cache_map(&plan->tmv, a->v_cache, rows, plan->desc.kv_dtype, plan->desc.page_size)) {
      plan->tk = plan->tv = nullptr;
      plan->tpages = -1;
      return PA_ERR_CUDA;
    }
    plan->tk = a->k_cache;
    plan->tv = a->v_cache;
    plan->tpages = a->num_pages;
  }
  k->tm_k = plan->tmk;
  k->tm_v = plan->tmv;
  return PA_OK;
}

template <int KVT, int SM, bool DUMP>
cudaError_t launch_t(const pa::KParams &k, size_t smem, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(k.grid);
  cfg.blockDim = dim3(pa::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa::decode_kernel<KVT, SM, DUMP>, k);
}

template <int SM>
cudaError_t launch_umma(const pa::KParams &k, size_t smem, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(k.grid);
  cfg.blockDim = dim3(pa::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  pa::KParams ku = k;
  // The tcgen05 kernel folds the per-token V scale into P relative to its maximum and
  // undoes the 256 of P's range itself: only the scalar V scale is left for the end
  // (without the mma.sync kernel's 2^-8).
  if (SM == PA_SCALE_PER_TOKEN) ku.vpost = 1.f;
  if (SM == PA_SCALE_SCALAR) ku.vpost = k.vpost * 256.f;
  return cudaLaunchKernelEx(&cfg, pa::decode_umma_kernel<SM>, ku);
}

template <bool DUMP>
cudaError_t launch(const pa_plan_desc_t &d, const pa::KParams &k, size_t smem, cudaStream_t s) {
  const bool pdl = (d.flags & PA_PLAN_NO_PDL) == 0;
  if (!DUMP && use_umma(d)) {
    if (d.scale_mode == PA_SCALE_SCALAR) return launch_umma<PA_SCALE_SCALAR>(k, smem, s, pdl);
    return launch_umma<PA_SCALE_PER_TOKEN>(k, smem, s, pdl);
  }
  if (d.kv_dtype == PA_KV_BF16) return launch_t<PA_KV_BF16, PA_SCALE_NONE, DUMP>(k, smem, s, pdl);
  if (d.scale_mode == PA_SCALE_SCALAR)
    return launch_t<PA_KV_FP8_E4M3, PA_SCALE_SCALAR, DUMP>(k, smem, s, pdl);
  return launch_t<PA_KV_FP8_E4M3, PA_SCALE_PER_TOKEN, DUMP>(k, smem, s, pdl);
}

// After pa_decode_check has passed: kernel parameters for a launch.
pa_status_t prepare_call(pa_plan *plan, const pa_decode_args_t *a, pa::KParams *k) {
  if (plan->ws == nullptr) return PA_ERR_WORKSPACE;
  fill_params(plan, a, k);
  return tensor_maps(plan, a, k);
}

size_t gather_tile_bytes(const pa_plan_desc_t &d) {
  return d.kv_dtype == PA_KV_FP8_E4M3 ? (size_t)(pa::kDumpHeader + 2 * pa::kTile * pa::kD + 1024)
                                      : (size_t)(pa::kDumpHeader + 4 * pa::kTile * pa::kD);
}

}  // namespace

extern "C" {

const char *pa_status_string(pa_status_t s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CAPACITY: return "PA_ERR_CAPACITY";
    case PA_ERR_RAGGED: return "PA_ERR_RAGGED";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_DATA: return "PA_ERR_DEVICE_DATA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
  }
  return "PA_ERR_UNKNOWN";
}

pa_status_t pa_plan_validate(const pa_plan_desc_t *desc) { return validate(desc); }

size_t pa_plan_workspace_size(const pa_plan_desc_t *desc) {
  Geometry g;
  return geometry(desc, &g) == PA_OK ? g.ws : 0;
}

pa_status_t pa_plan_create(const pa_plan_desc_t *desc, void *d_workspace, size_t workspace_bytes,
                           pa_plan_t **plan) {
  if (plan == nullptr) return PA_ERR_INVALID_ARG;
  *plan = nullptr;
  Geometry g;
  pa_status_t st = geometry(desc, &g);
  if (st != PA_OK) return st;
  int dev = -1;
  if (d_workspace == nullptr && workspace_bytes == 0) {
    // Check-only plan: validates calls with pa_decode_check, never launches.
  } else {
    if (d_workspace == nullptr || !aligned(d_workspace, 256) || workspace_bytes < g.ws)
      return PA_ERR_WORKSPACE;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemset(d_workspace, 0, g.off_ml) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
    // Raise the kernels' dynamic shared-memory limit to the device maximum (not to this
    // plan's carve), so that plans of different sizes never lower it under each other.
    int smem_optin = 0;
    if (cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        (size_t)smem_optin < g.smem)
      return PA_ERR_UNSUPPORTED;
    if (prepare_kernels(*desc, (size_t)smem_optin) != cudaSuccess) return PA_ERR_CUDA;
  }
  pa_plan *p = new (std::nothrow) pa_plan;
  if (p == nullptr) return PA_ERR_INVALID_ARG;
  p->desc = *desc;
  p->geo = g;
  p->device = dev;
  p->ws = d_workspace;
  *plan = p;
  return PA_OK;
}

pa_status_t pa_decode_check(const pa_plan_t *plan, const pa_decode_args_t *a) {
  if (plan == nullptr || a == nullptr) return PA_ERR_INVALID_ARG;
  const pa_plan_desc_t &d = plan->desc;
  if (a->reserved0 != 0) return PA_ERR_INVALID_ARG;
  if (a->num_seqs < 0 || a->num_rows < 0) return PA_ERR_INVALID_ARG;
  if (a->num_seqs > d.max_batch || a->num_rows > d.max_rows) return PA_ERR_CAPACITY;
  if (a->num_seqs == 0) return a->num_rows == 0 ? PA_OK : PA_ERR_RAGGED;
  if (a->k_cache == nullptr || a->v_cache == nullptr || a->block_table == nullptr ||
      a->context_lens == nullptr || a->out == nullptr || (a->num_rows > 0 && a->q == nullptr))
    return PA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) ||
      !aligned(a->out, 16) || !aligned(a->lse, 4) || !aligned(a->block_table, 4) ||
      !aligned(a->context_lens, 4))
    return PA_ERR_ALIGN;
  if (d.scale_mode == PA_SCALE_PER_TOKEN) {
    if (a->k_scale == nullptr || a->v_scale == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned(a->k_scale, 16) || !aligned(a->v_scale, 16)) return PA_ERR_ALIGN;
  }
  if (d.scale_mode == PA_SCALE_SCALAR) {
    if (!std::isfinite(a->k_scale_scalar) || !std::isfinite(a->v_scale_scalar) ||
        a->k_scale_scalar < 0.f || a->v_scale_scalar < 0.f)
      return PA_ERR_INVALID_ARG;
  }
  if (!std::isfinite(a->sm_scale) || a->sm_scale <= 0.f) return PA_ERR_INVALID_ARG;
  if (a->block_table_stride < 1 || a->num_pages < 1) return PA_ERR_INVALID_ARG;
  if (a->num_pages * d.num_kv_heads * d.page_size > (int64_t)INT32_MAX) return PA_ERR_CAPACITY;
  const int B = a->num_seqs;
  if (d.q_mode == PA_Q_UNIFORM) {
    // A uniform plan must really see a uniform segment (ROCm/ATOM PR 2122, section 2).
    if ((int64_t)a->num_rows != (int64_t)B * d.q_len) return PA_ERR_RAGGED;
    if (a->cu_seqlens_q_host != nullptr)
      for (int r = 0; r <= B; ++r)
        if (a->cu_seqlens_q_host[r] != r * d.q_len) return PA_ERR_RAGGED;
    if (a->cu_seqlens_q != nullptr && !aligned(a->cu_seqlens_q, 4)) return PA_ERR_ALIGN;
  } else {
    if (a->cu_seqlens_q == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned(a->cu_seqlens_q, 4)) return PA_ERR_ALIGN;
    if (a->cu_seqlens_q_host != nullptr) {
      const int32_t *cu = a->cu_seqlens_q_host;
      if (cu[0] != 0 || cu[B] != a->num_rows) return PA_ERR_INVALID_ARG;
      for (int r = 0; r < B; ++r) {
        const int ql = cu[r + 1] - cu[r];
        if (ql < 0) return PA_ERR_INVALID_ARG;
        if (ql > d.q_len) return PA_ERR_CAPACITY;
      }
    }
  }
  if (a->selected_pages != nullptr) {
    if (d.max_selected_pages == 0) return PA_ERR_UNSUPPORTED;
    if (a->num_selected == nullptr) return PA_ERR_INVALID_ARG;
    if (a->selected_stride < 1) return PA_ERR_INVALID_ARG;
    if (a->selected_stride > d.max_selected_pages) return PA_ERR_CAPACITY;
    if (!aligned(a->selected_pages, 4) || !aligned(a->num_selected, 4)) return PA_ERR_ALIGN;
  }
  return PA_OK;
}

pa_status_t pa_decode(pa_plan_t *plan, const pa_decode_args_t *args, void *stream) {
  pa::KParams k;
  std::memset(&k, 0, sizeof(k));
  pa_status_t st = pa_decode_check(plan, args);
  if (st != PA_OK) return st;
  if (args->num_seqs == 0) return PA_OK;
  if ((st = prepare_call(plan, args, &k)) != PA_OK) return st;
  if (launch<false>(plan->desc, k, plan->geo.smem, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_plan_get_device_status(pa_plan_t *plan, uint32_t *flags, int clear) {
  if (plan == nullptr || flags == nullptr) return PA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  uint32_t *st = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(plan->ws) + plan->geo.off_status);
  if (cudaMemcpy(flags, st, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (clear && cudaMemset(st, 0, sizeof(uint32_t)) != cudaSuccess) return PA_ERR_CUDA;
  if (clear && cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_plan_get_info(const pa_plan_t *plan, pa_plan_info_t *info) {
  if (plan == nullptr || info == nullptr) return PA_ERR_INVALID_ARG;
  info->grid_ctas = plan->geo.grid;
  info->stages = plan->geo.nstage;
  info->threads_per_cta = pa::kThreads;
  info->tile_tokens = pa::kTile;
  info->smem_bytes = (int64_t)plan->geo.smem;
  info->workspace_bytes = (int64_t)plan->geo.ws;
  info->partial_slots = plan->geo.slots;
  info->kernel = use_umma(plan->desc) ? 1 : 0;
  info->reserved = 0;
  return PA_OK;
}

void pa_plan_destroy(pa_plan_t *plan) { delete plan; }

pa_status_t pa_debug_row_map(pa_plan_t *plan, const pa_decode_args_t *args, int32_t *row_map,
                             void *stream) {
  if (row_map == nullptr || !aligned(row_map, 4)) return PA_ERR_INVALID_ARG;
  pa::KParams k;
  std::memset(&k, 0, sizeof(k));
  pa_status_t st = pa_decode_check(plan, args);
  if (st != PA_OK) return st;
  if (args->num_seqs == 0) return PA_OK;
  if (plan->ws == nullptr) return PA_ERR_WORKSPACE;
  fill_params(plan, args, &k);
  const int blocks = (args->num_seqs + 127) / 128;
  (void)cudaGetLastError();  // drop an earlier, unrelated launch error
  pa::row_map_kernel<<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(k, row_map);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_debug_gather_tile_bytes(const pa_plan_t *plan) {
  return plan ? gather_tile_bytes(plan->desc) : 0;
}

pa_status_t pa_debug_gather(pa_plan_t *plan, const pa_decode_args_t *args, void *dump,
                            size_t dump_bytes, void *stream) {
  if (dump == nullptr || !aligned(dump, 16)) return PA_ERR_INVALID_ARG;
  pa::KParams k;
  std::memset(&k, 0, sizeof(k));
  pa_status_t st = pa_decode_check(plan, args);
  if (st != PA_OK) return st;
  if (args->num_seqs == 0) return PA_OK;
  if ((st = prepare_call(plan, args, &k)) != PA_OK) return st;
  k.dump = static_cast<uint8_t *>(dump);
  k.dump_tiles = (int64_t)(dump_bytes / gather_tile_bytes(plan->desc));
  if (launch<true>(plan->desc, k, plan->geo.smem, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// Decode without a caller-provided workspace.  The split-K scratch (status word, arrival
// counters, partial maxima, sums and accumulators) lives in one fixed device array that
// this library defines; every GPU that loads the library holds it until the process
// exits.  See pa_decode_noalloc in pa.h.

namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  std::once_flag once;
  void *ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Once per device, with that device current: the device address of the scratch array
// (its name in host code is only a stand-in) and the kernels' shared-memory limit.
void noalloc_setup(NoAllocDevice &nd) {
  void *ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  int dev = 0, smem_optin = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  pa_plan_desc_t d;
  std::memset(&d, 0, sizeof(d));
  const int modes[3][2] = {{PA_KV_FP8_E4M3, PA_SCALE_PER_TOKEN},
                           {PA_KV_FP8_E4M3, PA_SCALE_SCALAR},
                           {PA_KV_BF16, PA_SCALE_NONE}};
  for (int m = 0; m < 3 && e == cudaSuccess; ++m) {
    d.kv_dtype = modes[m][0];
    d.scale_mode = modes[m][1];
    // q_len 1 with the tcgen05 flag raises the tcgen05 kernels' limit too (for FP8 modes)
    d.q_len = 1;
    d.flags = PA_PLAN_TCGEN05;
    e = prepare_kernels(d, (size_t)smem_optin);
  }
  nd.ptr = ptr;
  nd.err = e;
}

}  // namespace

extern "C" pa_status_t pa_decode_noalloc(const pa_plan_desc_t *desc, const pa_decode_args_t *args,
                                         void *stream) {
  if (desc == nullptr || args == nullptr) return PA_ERR_INVALID_ARG;
  Geometry g;
  pa_status_t st = geometry(desc, &g);
  if (st != PA_OK) return st;
  if (g.ws > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_CAPACITY;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PA_ERR_UNSUPPORTED;
  NoAllocDevice &nd = g_noalloc_dev[dev];
  std::call_once(nd.once, noalloc_setup, std::ref(nd));
  if (nd.err != cudaSuccess || nd.ptr == nullptr) return PA_ERR_CUDA;

  pa_plan plan;  // on the stack: no host or device allocation
  plan.desc = *desc;
  plan.geo = g;
  plan.device = dev;
  plan.ws = nd.ptr;
  if ((st = pa_decode_check(&plan, args)) != PA_OK) return st;
  if (args->num_seqs == 0) return PA_OK;
  // The status word and the arrival counters must start at zero; the rest of the
  // scratch is written before it is read.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(nd.ptr, 0, g.off_ml, s) != cudaSuccess) return PA_ERR_CUDA;
  pa::KParams k;
  std::memset(&k, 0, sizeof(k));
  if ((st = prepare_call(&plan, args, &k)) != PA_OK) return st;
  if (launch<false>(plan.desc, k, g.smem, s) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

extern "C" pa_status_t pa_debug_trace(void *host, size_t bytes) {
#ifdef PA_TRACE
  if (host == nullptr) return PA_ERR_INVALID_ARG;
  const size_t n = bytes < sizeof(pa::g_trace) ? bytes : sizeof(pa::g_trace);
  return cudaMemcpyFromSymbol(host, pa::g_trace, n) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
#else
  (void)host;
  (void)bytes;
  return PA_ERR_UNSUPPORTED;
#endif
}
