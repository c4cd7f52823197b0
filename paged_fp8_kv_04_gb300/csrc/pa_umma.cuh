// pa_umma.cuh -- paged FP8 decode on the tcgen05 tensor cores (one query token per
// request: the 16 query heads of a KV head form one 16-row group).
//
// Per 128-token tile of one (request, KV head):
//   S^T[tok][n] = K[tok][:] . Q[n][:]    tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 16
//                                        heads, A = the K tile exactly as TMA left it
//                                        (K-major, 128-byte swizzle), B = the query as an
//                                        exact e4m3 hi + lo pair (two MMAs into one S).
//   softmax                              TMEM lane = token; the two warps of a lane quarter
//                                        take 8 heads each: per-token K scale folded into
//                                        the score, causal / page mask, a running maximum
//                                        per (warp slice, head) by warp reduction, exp2.
//   O_w^T[d][n] = V^T[d][tok] . P^T      kind::f8f6f4 again, M = 128 head_dim lanes, N = 16,
//                                        A = the V tile as TMA left it (MN-major), B = P as
//                                        e4m3 hi + lo with the per-token V scale folded in,
//                                        relative to the slice's largest p * v_scale per
//                                        head; one O tile per 32-token slice.
//   O update                             TMEM lane = head_dim: o = o * alpha + O_w * beta in
//                                        fp32 registers, one tile late so that it overlaps
//                                        the next tile's softmax and the PV in flight.
// Neither K nor V is widened on the SM sub-partitions; the tensor core reads the cache
// bytes.  P is carried with 8 significant bits (hi + lo) relative to the largest
// p * v_scale of its own 32 tokens, so a tile's small probabilities are not flushed however
// far below the running maximum the tile lies, nor a token's weight by a neighbour's
// larger V scale; what a tile can lose is below 2^-18 of its largest weighted term.
//
// Warp roles (384 threads): warps 0-7 run the softmax on every tile (warp w: token slice
// w & 3, heads 8 (w >> 2) .. + 7); warp 8 is the TMA producer (the same page gather as the
// mma.sync kernel); warp 9 converts queries and issues QK^T up to four tiles ahead; warp
// 10 issues PV as soon as a tile's P is published; warp 11 only gives back registers.
// Every wait is bounded; TMEM is released on every path.
#pragma once

#include "pa_consumer.cuh"
#include "pa_producer.cuh"

namespace pa {

// Offsets in the shared merge region (Smem::merge()), which this kernel uses instead of
// the mma.sync kernel's token-slice exchange.
constexpr int kUQ = 0;        // query hi / lo, 2 slots x 4096: hi at +0, lo at +2048 (SW128)
constexpr int kUP = 8192;     // P^T of tile parity b at +4096 b: hi at +0, lo at +2048 ([tok][16 B])
constexpr int kUAB = 16384;   // alpha [3 tiles][4 slices][16 heads] f32; beta at +768
constexpr int kUML = 17920;   // per-slice m [2 sequences][4][16] f32 (+1024 per parity); l at +512
constexpr int kUKF = 19968;   // kfold * 2^-sigma of each query slot [2] f32
static_assert(kUKF + 8 <= kMergeBytes, "tcgen05 kernel scratch must fit the merge region");

// TMEM columns: S of tile i at 16 (i & 3); O tiles of tile parity b at 64 + 64 b + 16 * slice.
constexpr uint32_t kTmemCols = 256;
constexpr int kSBufs = 4;

// S has four buffers, released by s_free once every softmax warp has loaded it.  PV of
// tile i + 2 is issued only after every softmax warp has published P of tile i + 2, which
// it does after the O update of tile i + 1, itself after waiting for PV of tile i + 1 and
// after the update of tile i: so P and the O tiles need two buffers and alpha / beta three.
struct UBars {
  uint32_t s_full[kSBufs], s_free[kSBufs], p_ready[2], o_full[2], qready[2], qfree[2];
  uint32_t tdone, mmadone;
};

__device__ __forceinline__ UBars ubars(const Smem &sm) {
  const uint32_t b = sm.bar0 + 8 * (2 * sm.nstage + 3);
  UBars u;
#pragma unroll
  for (int k = 0; k < kSBufs; ++k) {
    u.s_full[k] = b + 8 * k;
    u.s_free[k] = b + 32 + 8 * k;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    u.p_ready[k] = b + 64 + 8 * k;
    u.o_full[k] = b + 80 + 8 * k;
    u.qready[k] = b + 96 + 8 * k;
    u.qfree[k] = b + 112 + 8 * k;
  }
  u.tdone = b + 128;
  u.mmadone = b + 136;
  return u;
}

static_assert(2 * kSBufs + 10 <= kUmmaBars, "the tcgen05 kernel's barriers must fit their slots");

__device__ __forceinline__ void umma_init_bars(const UBars &u) {
#pragma unroll
  for (int k = 0; k < kSBufs; ++k) {
    mbar_init(u.s_full[k], 1);      // tcgen05.commit after QK^T into S buffer k
    mbar_init(u.s_free[k], kNCW);   // every softmax warp has loaded S buffer k
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    mbar_init(u.p_ready[k], kNCW);  // every softmax warp has written its P, alpha, beta
    mbar_init(u.o_full[k], 1);      // tcgen05.commit after PV
    mbar_init(u.qready[k], 1);      // the MMA warp has converted a query
    mbar_init(u.qfree[k], kNCW);    // every softmax warp has read that query's scale
  }
  mbar_init(u.tdone, kNCW);         // softmax warps are done with TMEM
  mbar_init(u.mmadone, 2);          // every MMA of both issuing warps has completed
}

// ----------------------------------------------------------------------- the MMA warp

// The request's query (16 heads x 128 bf16 in the raw slot at `raw`) as e4m3 hi and lo
// parts at scale 2^sigma, which puts the group's largest magnitude in [128, 256).  A
// bf16 value has 8 significant bits and an e4m3 code 4, so the rounding residual of the
// hi part is itself an e4m3 code for every element at or above 2^-10 of that magnitude
// (smaller ones keep an absolute error below 2^-18 of it).  Written K-major with the
// 128-byte swizzle: row n, 16-byte chunk c at chunk c ^ (n & 7).  Returns kfold/2^sigma.
__device__ float umma_convert_query(const KParams &p, uint32_t raw, uint32_t qhl, int lane) {
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int u = lane + 32 * k, n = u >> 3, c = u & 7;
    const uint4 x = lds128(raw + n * (kD * 2) + c * 32), y = lds128(raw + n * (kD * 2) + c * 32 + 16);
    const uint32_t wd[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(wd[j])), fabsf(bf16hi(wd[j]))));
  }
  const uint32_t ab = __reduce_max_sync(~0u, __float_as_uint(amax));
  if (ab >= 0x7F800000u && lane == 0) atomicOr(p.status, PA_DEV_Q_RANGE);
  int sig = 0;
  if (ab != 0u) sig = min(max(7 - ((int)(ab >> 23) - 127), -126), 126);
  const float up = __uint_as_float((uint32_t)(sig + 127) << 23);
#pragma unroll 1
  for (int k = 0; k < 4; ++k) {
    const int u = lane + 32 * k, n = u >> 3, c = u & 7;
    const uint4 x = lds128(raw + n * (kD * 2) + c * 32), y = lds128(raw + n * (kD * 2) + c * 32 + 16);
    const uint32_t wd[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
    uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // word j: d = 16 c + 2 j, + 1
      const float y0 = bf16lo(wd[j]) * up, y1 = bf16hi(wd[j]) * up;
      const uint32_t hc = pack_e4m3x2(y0, y1);
      float h0, h1;
      e4m3x2_to_f32x2(hc, h0, h1);
      const uint32_t lc = pack_e4m3x2(y0 - h0, y1 - h1);
      hw[j >> 1] |= hc << (16 * (j & 1));
      lw[j >> 1] |= lc << (16 * (j & 1));
    }
    const uint32_t off = n * 128 + ((c ^ (n & 7)) << 4);
    sts128(qhl + off, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(qhl + 2048 + off, make_uint4(lw[0], lw[1], lw[2], lw[3]));
  }
  return p.kfold * __uint_as_float((uint32_t)(127 - sig) << 23);
}

// Warp 9: queries and QK^T.  Tile j's scores go to S buffer j & 3 as soon as its stage
// has landed and the buffer's previous scores (tile j - 4) have been loaded.
__device__ void run_qk_warp(const KParams &p, const Smem &sm, const UBars &ub, int a, int b,
                            uint32_t tm) {
  const int lane = threadIdx.x & 31;
  const int n = b - a;
  const uint32_t ua = sm.merge();
  constexpr uint32_t idq = umma_idesc_e4m3(128, 16, 0, 0);  // K-major A and B
  int seg = 0, qb = 0;
  bool ok = true;
  for (int j = 0; j < n && ok; ++j) {
    const int s = j % p.nstage;
    if (!mbar_wait_bounded(sm.full(s), (j / p.nstage) & 1)) {
      ok = false;
      break;
    }
    const StageMeta *mt = sm.meta(s);
    if (mt->flags & F_BEGIN) {
      qb = seg & 1;
      const int use = seg >> 1;
      ++seg;
      // every softmax warp has read the scale of the request that used this slot before
      if (use >= 1 && !mbar_wait_bounded(ub.qfree[qb], (use - 1) & 1)) {
        ok = false;
        break;
      }
      const float kf = umma_convert_query(p, sm.qslot(mt->qslot), ua + kUQ + qb * 4096, lane);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(ua + kUKF + 4 * qb), "f"(kf) : "memory");
        mbar_arrive(sm.qempty(mt->qslot));
        mbar_arrive(ub.qready[qb]);
      }
    }
    const int sb = j & (kSBufs - 1);
    if (j >= kSBufs && !mbar_wait_bounded(ub.s_free[sb], ((j - kSBufs) / kSBufs) & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (lane == 0) {
      const uint32_t st = sm.stage(s), q = ua + kUQ + qb * 4096;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ka = umma_sdesc(st + 32 * k, 1024, 1024, 2);
        umma_e4m3(tm + 16 * sb, ka, umma_sdesc(q + 32 * k, 1024, 1024, 2), idq, k > 0 ? 1u : 0u);
        umma_e4m3(tm + 16 * sb, ka, umma_sdesc(q + 2048 + 32 * k, 1024, 1024, 2), idq, 1u);
      }
      umma_commit(ub.s_full[sb]);
    }
    __syncwarp();
  }
  if (!ok && lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
  if (lane == 0) umma_commit(ub.mmadone);
  __syncwarp();
}

// Warp 10: PV of tile i as soon as every softmax warp has published its P.  Stage s of
// tile i is released by a commit after the PV (its QK^T completed before P existed).
__device__ void run_pv_warp(const KParams &p, const Smem &sm, const UBars &ub, int a, int b,
                            uint32_t tm) {
  const int lane = threadIdx.x & 31;
  const int n = b - a;
  const uint32_t ua = sm.merge();
  constexpr uint32_t idp = umma_idesc_e4m3(128, 16, 1, 1);  // MN-major A (V^T) and B (P^T)
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    const int s = i % p.nstage, w = i & 1;
    if (!mbar_wait_bounded(ub.p_ready[w], (i >> 1) & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (lane == 0) {
      const uint32_t v = sm.stage(s) + 16384, pt = ua + kUP + w * 4096;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // token slice ks = the 32 tokens of softmax warps ks, ks + 4
        const uint32_t d = tm + 64 + 64 * w + 16 * ks;
        const uint64_t va = umma_sdesc(v + 4096 * ks, 1024, 1024, 2);
        umma_e4m3(d, va, umma_sdesc(pt + 512 * ks, 128, 128, 0), idp, 0u);
        umma_e4m3(d, va, umma_sdesc(pt + 2048 + 512 * ks, 128, 128, 0), idp, 1u);
      }
      umma_commit(ub.o_full[w]);
      umma_commit(sm.empty(s));
    }
    __syncwarp();
  }
  if (!ok && lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
  if (lane == 0) umma_commit(ub.mmadone);
  __syncwarp();
}

// ------------------------------------------------------------- split-K partial merge

// The last CTA to finish a split sequence merges every partial ([slot][16 heads][128]
// unnormalised fp32 and (m, l) per head): thread u takes (head, 4 head_dim) units and
// brings up to 8 partials per round with independent loads.
__device__ void umma_merge_partials(const KParams &p, int h, int row0, int c_first, int n,
                                    int ctid) {
  const int Hq = p.Hkv * kG;
  const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml);
  const float4 *src = reinterpret_cast<const float4 *>(p.part_o);
  for (int u = ctid; u < kG * 32; u += kNCW * 32) {
    const int row = u >> 5, d4 = u & 31;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < n; k0 += 8) {
      float2 mlv[8];
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (k0 + j < n) {
          const int64_t sl = slot_of(c_first + k0 + j, c_first);
          mlv[j] = __ldcg(ml + sl * p.mmax + row);
          v[j] = __ldcg(src + (sl * p.mmax + row) * 32 + d4);
        } else {
          mlv[j] = make_float2(-INFINITY, 0.f);
          v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float nm = M;
#pragma unroll
      for (int j = 0; j < 8; ++j) nm = fmaxf(nm, mlv[j].x);
      if (nm == -INFINITY) continue;
      const float c = fast_exp2(M - nm);
      acc.x *= c;
      acc.y *= c;
      acc.z *= c;
      acc.w *= c;
      L *= c;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wgt = fast_exp2(mlv[j].x - nm);
        acc.x += wgt * v[j].x;
        acc.y += wgt * v[j].y;
        acc.z += wgt * v[j].z;
        acc.w += wgt * v[j].w;
        L += wgt * mlv[j].y;
      }
      M = nm;
    }
    const float sc = L > 0.f ? p.vpost / L : 0.f;
    const float vv[4] = {acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc};
    store_out(p, ((int64_t)row0 * Hq + h * kG + row) * kD + 4 * d4, vv, 4);
    if (d4 == 0 && p.lse != nullptr)
      p.lse[(int64_t)row0 * Hq + h * kG + row] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------- softmax warps

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}

// e4m3 hi part of y in [0, 256]: y rounded to 4 significant bits.  At or above 2^-6 that
// is an e4m3 normal whose code is read off the fp32 bits (exponent rebias 127 -> 7); below
// it the hi part is 0 and the lo part carries y.
__device__ __forceinline__ float hi_e4m3(float y, uint32_t &code) {
  const uint32_t u = (__float_as_uint(y) + 0x80000u) & 0xFFF00000u;
  const bool nz = u >= 0x3C800000u;  // 2^-6
  code = nz ? (u >> 20) - 960u : 0u;
  return nz ? __uint_as_float(u) : 0.f;
}

template <int SM>
__device__ void run_softmax(const KParams &p, const Smem &sm, const UBars &ub, int a, int b,
                            uint32_t tm, int warp, int lane) {
  const int q = warp & 3, hh = warp >> 2;  // token slice (TMEM lane quarter), head half
  const int t = 32 * q + lane;             // token of a tile (S lanes), head_dim d (O lanes)
  const int ctid = warp * 32 + lane;
  const uint32_t ua = sm.merge();
  const uint32_t tl = tm + ((uint32_t)(32 * q) << 16);
  const int Hq = p.Hkv * kG;
  const int32_t *tstart = sm.tstart();
  uint32_t cphase = 0;

  // Requests without tiles (empty key set for every row): zero rows, lse = -inf.
  for (int r = blockIdx.x; r < p.num_seqs; r += gridDim.x) {
    if (tstart[r + 1] != tstart[r]) continue;
    uint32_t fl = 0;
    const ReqInfo ri = request_info(p, r, fl);
    if (ri.qlen <= 0) continue;
    const int64_t e0 = (int64_t)ri.row0 * Hq * kD, ne = (int64_t)ri.qlen * Hq * kD;
    const float z[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t e = 4 * ctid; e < ne; e += 4 * kNCW * 32) store_out(p, e0 + e, z, 4);
    if (p.lse != nullptr)
      for (int e = ctid; e < ri.qlen * Hq; e += kNCW * 32) p.lse[(int64_t)ri.row0 * Hq + e] = -INFINITY;
  }

  float o[4][8];  // head_dim t of heads 8 hh .. 8 hh + 7, per token slice
  float mr[8];    // running maximum of this warp's (slice, head) pairs (log2 units)
  float l[8];     // this token's sums per head, relative to mr
  float kf = 0.f;
  int seg = 0, nseq = 0, pend = -1;
  bool has_head = false, has_tail = false, ok = true;

  // The O tiles of tile j (whose PV is in flight): wait for them and start their loads.
  uint32_t ot[4][8];
  auto load_o = [&](int j) -> bool {
    if (!mbar_wait_bounded(ub.o_full[j & 1], (j >> 1) & 1)) return false;
    tc_fence_after();
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) tmem_ld8_async(tl + 64 + 64 * (j & 1) + 16 * sl + 8 * hh, ot[sl]);
    return true;
  };
  // o = o * alpha + O_tile * beta (the loads of load_o have completed).
  auto update = [&](int j) {
    const uint32_t ab = ua + kUAB + (j % 3) * 256 + 32 * hh;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      const uint4 a0 = lds128(ab + 64 * sl), a1 = lds128(ab + 64 * sl + 16);
      const uint4 b0 = lds128(ab + 768 + 64 * sl), b1 = lds128(ab + 768 + 64 * sl + 16);
      const uint32_t al[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint32_t be[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k)
        o[sl][k] = fmaf(o[sl][k], __uint_as_float(al[k]),
                        __uint_as_float(ot[sl][k]) * __uint_as_float(be[k]));
    }
  };

  const int n = b - a;
  for (int i = 0; i < n && ok; ++i) {
    const int s = i % p.nstage;
    if (!mbar_wait_bounded(sm.full(s), (i / p.nstage) & 1)) {
      ok = false;
      break;
    }
    const StageMeta *mt = sm.meta(s);
    const int flags = mt->flags, r = mt->r, h = mt->h, L = mt->L, row0 = mt->row0;
    if (flags & F_BEGIN) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        mr[k] = -INFINITY;
        l[k] = 0.f;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) o[sl][k] = 0.f;
      }
      const int qb = seg & 1, use = seg >> 1;
      ++seg;
      if (!mbar_wait_bounded(ub.qready[qb], use & 1)) {
        ok = false;
        break;
      }
      kf = lds_f32(ua + kUKF + 4 * qb);
      __syncwarp();
      if (lane == 0) mbar_arrive(ub.qfree[qb]);
    }
    const uint32_t st = sm.stage(s);

    // ---- scores of token t against heads 8 hh .. 8 hh + 7
    const int sb = i & (kSBufs - 1);
    if (!mbar_wait_bounded(ub.s_full[sb], (i / kSBufs) & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t xr[8];
    tmem_ld8_async(tl + 16 * sb + 8 * hh, xr);
    tmem_wait8(xr);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(ub.s_free[sb]);
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = __uint_as_float(xr[k]);
    float ks = 1.f, vs = 1.f;
    if (SM == PA_SCALE_PER_TOKEN) {
      ks = lds_f32(st + 32768 + 4 * t);
      vs = lds_f32(st + 33280 + 4 * t);
    }
    const float c = ks * kf;
    bool masked = false;
    if (flags & F_MASK) {
      const int pp = mt->page_pos[t >> p.ps_shift];
      const int pos = pp < 0 ? -1 : pp + (t & (p.ps - 1));
      masked = pos < 0 || pos >= L;  // one query token: the cutoff is L
    }
    // a masked slot's scales may be stale shared memory (an empty page slot), NaN included
    if (masked) vs = 0.f;
    float alpha[8], gam[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[k] = masked ? -INFINITY : x[k] * c;
      const float tmx = warp_max_f32(x[k]);
      const float mn = fmaxf(mr[k], tmx);
      alpha[k] = (mn == mr[k]) ? 1.f : fast_exp2(mr[k] - mn);
      gam[k] = (tmx == -INFINITY) ? 0.f : fast_exp2(tmx - mn);
      mr[k] = mn;
      x[k] = fast_exp2(x[k] - (tmx == -INFINITY ? 0.f : tmx));  // p relative to the tile max
    }
    // per head, W = the slice's largest p * v_scale: the largest product, not the largest
    // scale, so that a token with p = 1 and a small scale keeps its 8 bits next to a token
    // with a large scale and p ~ 0
    // with a power of two F = 2^(7 - floor(log2 W)) (at most 2^120): P' = p * v_scale * F
    // <= 256, and the O tile is scaled back by 1 / F
    float xv[8], F[8], Fi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (SM == PA_SCALE_PER_TOKEN) {
        xv[k] = x[k] * vs;
        const float W = warp_max_f32(xv[k]);
        const int ew = (int)((__float_as_uint(W) >> 23) & 0xFFu) - 127;
        const int ef = min(7 - ew, 120);
        F[k] = W > 0.f ? __uint_as_float((uint32_t)(ef + 127) << 23) : 0.f;
        Fi[k] = W > 0.f ? __uint_as_float((uint32_t)(127 - ef) << 23) : 0.f;
      } else {
        xv[k] = x[k];
        F[k] = 256.f;
        Fi[k] = 1.f / 256.f;
      }
    }
    // ---- P' = p * v_scale * F as e4m3 hi + lo; running sums
    uint32_t hw[2] = {0u, 0u}, lw[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k0 = 2 * j, k1 = 2 * j + 1;
      l[k0] = fmaf(l[k0], alpha[k0], x[k0] * gam[k0]);
      l[k1] = fmaf(l[k1], alpha[k1], x[k1] * gam[k1]);
      const float y0 = xv[k0] * F[k0], y1 = xv[k1] * F[k1];
      uint32_t c0, c1;
      const float h0 = hi_e4m3(y0, c0), h1 = hi_e4m3(y1, c1);
      hw[j >> 1] |= (c0 | (c1 << 8)) << (16 * (j & 1));
      lw[j >> 1] |= pack_e4m3x2(y0 - h0, y1 - h1) << (16 * (j & 1));
    }
    // ---- the O update of the previous tile (its PV ran during this tile's softmax):
    // four TMEM loads in flight together, one wait
    if (pend >= 0) {
      if (!load_o(pend)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) tmem_wait8(ot[sl]);
      tc_fence_before();
      update(pend);
      pend = -1;
    }
    const uint32_t pt = ua + kUP + (i & 1) * 4096 + 16 * t + 8 * hh;
    sts64(pt, hw[0], hw[1]);
    sts64(pt + 2048, lw[0], lw[1]);
    {  // alpha (rescale of the slice's o) and beta (scale of its new O tile) per head
      const uint32_t ab = ua + kUAB + (i % 3) * 256 + 64 * q + 32 * hh;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (lane == k) {
          sts_f32(ab + 4 * k, alpha[k]);
          sts_f32(ab + 768 + 4 * k, gam[k] * Fi[k]);
        }
    }
    if (masked && hh == 0) {  // a masked slot's V bytes may be stale or NaN codes: 0 * NaN = NaN
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) sts128(st + 16384 + 128 * t + 16 * cc, make_uint4(0u, 0u, 0u, 0u));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(ub.p_ready[i & 1]);
      mbar_arrive(sm.empty(s));  // the stage is released once the PV commit also arrives
    }
    pend = i;
    if (!(flags & F_END)) continue;

    // ---- end of this CTA's part of sequence (r, h) --------------------------------------
    if (!load_o(i)) {
      ok = false;
      break;
    }
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) tmem_wait8(ot[sl]);
    tc_fence_before();
    update(i);
    pend = -1;
    const uint32_t mlb = ua + kUML + (nseq & 1) * 1024;
    ++nseq;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float v = l[k];
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(~0u, v, o2);
      if (lane == k) {
        sts_f32(mlb + (q * 16 + 8 * hh + k) * 4, mr[k]);
        sts_f32(mlb + 512 + (q * 16 + 8 * hh + k) * 4, v);
      }
    }
    cons_sync(p, sm, cphase);
    const bool whole = (flags & F_WHOLE) != 0;
    int slot = 0, c_first = 0, nc = 1;
    if (!whole) {
      const int nt = tstart[r + 1] - tstart[r];
      const int gs = tstart[r] * p.Hkv + h * nt;
      seq_ctas(p, tstart, r, h, gs, gs + nt, c_first, nc);
      slot = slot_of(sm.misc()[M_VCTA], c_first);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = 8 * hh + k;
      float ms[4], M = -INFINITY;
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        ms[sl] = lds_f32(mlb + (sl * 16 + row) * 4);
        M = fmaxf(M, ms[sl]);
      }
      float Ls = 0.f, of = 0.f;
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        const float f = ms[sl] == -INFINITY ? 0.f : fast_exp2(ms[sl] - M);
        Ls = fmaf(lds_f32(mlb + 512 + (sl * 16 + row) * 4), f, Ls);
        of = fmaf(o[sl][k], f, of);
      }
      if (whole) {
        const float v = Ls > 0.f ? of * (p.vpost / Ls) : 0.f;
        const int64_t e = ((int64_t)row0 * Hq + h * kG + row) * kD + t;
        if (p.out_f32)
          static_cast<float *>(p.out)[e] = v;
        else
          static_cast<__nv_bfloat16 *>(p.out)[e] = __float2bfloat16_rn(v);
        if (q == 0 && lane == k && p.lse != nullptr)
          p.lse[(int64_t)row0 * Hq + h * kG + row] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
      } else {
        __stcg(p.part_o + ((int64_t)slot * p.mmax + row) * kD + t, of);
        if (q == 0 && lane == k)
          __stcg(reinterpret_cast<float2 *>(p.part_ml) + (int64_t)slot * p.mmax + row, make_float2(M, Ls));
      }
    }
    if (whole) continue;
    // A split sequence: count this CTA's arrival; the last of the sequence's CTAs merges.
    const bool is_head = i < n - 1;
    __threadfence();
    cons_sync(p, sm, cphase);
    if (ctid == 0) {
      int32_t *rec = sm.misc() + (is_head ? M_HEAD : M_TAIL);
      rec[0] = r;
      rec[1] = h;
      rec[2] = row0;
      rec[3] = 1;
      rec[4] = c_first;
      rec[5] = nc;
      const int old = atomicAdd(p.counters + (r * p.Hkv + h), 1);
      sm.misc()[M_LAST + (is_head ? 0 : 1)] = (old == nc - 1) ? 1 : 0;
    }
    if (is_head)
      has_head = true;
    else
      has_tail = true;
  }
  if (!ok && lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
  // TMEM is no longer read by this warp
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(ub.tdone);
  if (!(has_head || has_tail)) return;
  cons_sync(p, sm, cphase);
#pragma unroll 1
  for (int k = 0; k < 2; ++k) {
    const bool mine_k = k == 0 ? has_head : has_tail;
    if (!mine_k || !sm.misc()[M_LAST + k]) continue;
    const int32_t *rec = sm.misc() + (k == 0 ? M_HEAD : M_TAIL);
    const int rr = rec[0], hh2 = rec[1];
    __threadfence();
    umma_merge_partials(p, hh2, rec[2], rec[4], rec[5], ctid);
    if (ctid == 0) p.counters[rr * p.Hkv + hh2] = 0;
  }
}

// ---------------------------------------------------------------------------- kernel

template <int SM>
__global__ void __launch_bounds__(kThreads, 1) decode_umma_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  const Smem sm = Smem::make(smem_raw + ((1024u - mis) & 1023u), p);
  const UBars ub = ubars(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), 1 + kNCW);  // the PV commit + every softmax warp
    }
    mbar_init(sm.qempty(0), 1);
    mbar_init(sm.qempty(1), 1);
    mbar_init(sm.consbar(), kNCW);
    umma_init_bars(ub);
    sm.misc()[M_ABORT] = 0;
    sm.misc()[M_LAST] = 0;
    sm.misc()[M_LAST + 1] = 0;
    sm.misc()[M_WCNT] = 0;
    fence_barrier_init();
  }
  if (warp == kNCW + 1) tmem_alloc(smem_u32(sm.misc() + M_TMEM), kTmemCols);
  tc_fence_before();
  pdl_launch_dependents();
  const uint32_t fl = scan_tiles(p, sm.tstart(), sm.misc() + M_WSUM);  // synchronises the CTA
  tc_fence_after();
  const uint32_t tm = (uint32_t)sm.misc()[M_TMEM];
  const uint32_t report = blockIdx.x == 0 ? fl : 0u;
  if (warp >= kNCW) {
    regs_dec<kProdRegs>();
    const int a = sm.misc()[M_WSUM], b = sm.misc()[M_WSUM + 1];
    if (warp == kNCW) {
      // The producer reads index inputs before the wait, q and the caches after it.
      if (a < b) run_producer<PA_KV_FP8_E4M3, SM>(p, sm, a, b, report);
      else {
        pdl_wait();
        if (report) atomicOr(p.status, report);
      }
    } else if (warp == kNCW + 1) {
      run_qk_warp(p, sm, ub, a, b, tm);
      // both issuers' MMAs have completed and the softmax warps are done with TMEM
      if (!mbar_wait_bounded(ub.mmadone, 0) && lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
      if (!mbar_wait_bounded(ub.tdone, 0) && lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
      tc_fence_after();
      tmem_dealloc(tm, kTmemCols);
    } else if (warp == kNCW + 2) {
      run_pv_warp(p, sm, ub, a, b, tm);
    }
    return;
  }
  regs_inc<kConsRegs>();
  const int a = sm.misc()[M_WSUM], b = sm.misc()[M_WSUM + 1];
  pdl_wait();  // softmax warps write outputs and the workspace
  if (report) atomicOr(p.status, report);
  run_softmax<SM>(p, sm, ub, a, b, tm, warp, lane);
}

}  // namespace pa
