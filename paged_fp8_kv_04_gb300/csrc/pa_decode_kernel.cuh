// pa_decode_kernel.cuh -- kernel entry points: decode, gather dump, row map.
#pragma once

#include "pa_consumer.cuh"
#include "pa_producer.cuh"

namespace pa {

// Copies one loaded stage to the gather dump (swizzle undone).  Header: 32 int32.
template <int KVT, int SM>
__device__ void dump_stage(const KParams &p, const Smem &sm, int s, int ctid, int tile_bytes) {
  const StageMeta *mt = sm.meta(s);
  const int gt = mt->gtile;
  if ((int64_t)gt >= p.dump_tiles) {
    if (ctid == 0) atomicOr(p.status, PA_DEV_DUMP_RANGE);
    return;
  }
  uint8_t *dst = p.dump + (int64_t)gt * tile_bytes;
  const int32_t *src_meta = reinterpret_cast<const int32_t *>(mt);
  if (ctid < 32) {
    int32_t v = 0;
    if (ctid < 24) v = src_meta[ctid];
    reinterpret_cast<int32_t *>(dst)[ctid] = v;
  }
  const uint32_t st = sm.stage(s);
  const int row_bytes = (KVT == PA_KV_FP8_E4M3) ? kD : 2 * kD;
  const int chunks = row_bytes / 16;  // 16-B chunks per token row
  uint8_t *kv = dst + kDumpHeader;
  for (int u = ctid; u < 2 * kTile * chunks; u += kNCW * 32) {
    const int which = u / (kTile * chunks);  // 0 = K, 1 = V
    const int rem = u - which * kTile * chunks;
    const int row = rem / chunks, cc = rem - row * chunks;
    uint32_t src;
    if (KVT == PA_KV_FP8_E4M3)
      src = st + which * 16384 + row * 128 + ((cc ^ (row & 7)) << 4);
    else
      src = st + which * 32768 + (cc >> 3) * 16384 + row * 128 + (((cc & 7) ^ (row & 7)) << 4);
    const uint4 v = lds128(src);
    *reinterpret_cast<uint4 *>(kv + which * kTile * row_bytes + row * row_bytes + cc * 16) = v;
  }
  if (KVT == PA_KV_FP8_E4M3 && SM == PA_SCALE_PER_TOKEN) {
    uint8_t *sc = kv + 2 * kTile * row_bytes;
    for (int u = ctid; u < 64; u += kNCW * 32)
      *reinterpret_cast<uint4 *>(sc + 16 * u) = lds128(st + 32768 + 16 * u);
  }
}

template <int KVT, int SM, bool DUMP>
__device__ void run_consumer(const KParams &p, const Smem &sm, int a, int b, int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int ctid = warp * 32 + lane;
  const int32_t *tstart = sm.tstart();
  uint32_t cphase = 0;

  // Requests without tiles (empty key set for every row): zero rows, lse = -inf.
  if (!DUMP) {
    const int Hq = p.Hkv * kG;
    for (int r = blockIdx.x; r < p.num_seqs; r += gridDim.x) {
      if (tstart[r + 1] != tstart[r]) continue;
      uint32_t fl = 0;
      const ReqInfo ri = request_info(p, r, fl);
      if (ri.qlen <= 0) continue;
      const int64_t e0 = (int64_t)ri.row0 * Hq * kD, n = (int64_t)ri.qlen * Hq * kD;
      const float z[4] = {0.f, 0.f, 0.f, 0.f};
      for (int64_t e = 4 * ctid; e < n; e += 4 * kNCW * 32) store_out(p, e0 + e, z, 4);
      if (p.lse != nullptr)
        for (int e = ctid; e < ri.qlen * Hq; e += kNCW * 32)
          p.lse[(int64_t)ri.row0 * Hq + e] = -INFINITY;
    }
  }
  if (a >= b) return;

  Frag f;
  reset_state(f);
  // Warp -> work map of the current request (fixed at its first tile):
  //  q_len <= 4: two groups of 4 warps take alternate tiles (warps 0-3 even, 4-7 odd);
  //              in a group, m-tile = query token, and 4 / q_len token slices per tile;
  //  q_len  > 4: every warp takes every tile, one m-tile (query token) per warp.
  int mt = 1, ts = 1, nsl = 1, mtile = 0, sub = 0, slice = 0, cut = 0;
  bool active = false, paired = true, quad = false;
  const int tile_bytes = (KVT == PA_KV_FP8_E4M3) ? (kDumpHeader + 2 * kTile * kD + 1024)
                                                  : (kDumpHeader + 4 * kTile * kD);
  const int n = b - a;
  bool has_head = false, has_tail = false;  // split sequences (records in misc[])
  if constexpr (DUMP) {
    // Gather test hook: every warp visits every tile.
    for (int i = 0; i < n; ++i) {
      const int s = i % p.nstage;
      if (!wait_tile(sm, s, (i / p.nstage) & 1, a + i)) {
        if (lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
        break;
      }
      const StageMeta *meta = sm.meta(s);
      if (meta->flags & F_BEGIN) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.qempty(meta->qslot));
      }
      dump_stage<KVT, SM>(p, sm, s, ctid, tile_bytes);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(s));
    }
    return;
  }

  // The CTA's tiles in order: (request r, KV head h, tile tj of nt), walked locally so
  // that a warp needs a stage only for the tiles it owns and for each request's first
  // tile (whose query every warp loads).  Stage arrivals: 1 per warp on a request's
  // first tile; otherwise the owners alone, weighted so that they count 8.
  int rw, hw, tjw;
  locate(tstart, p.num_seqs, p.Hkv, a, rw, hw, tjw);
  int ntw = tstart[rw + 1] - tstart[rw];
  int seg = 0, qlen = 1, row0 = 0, L = 0, mode = 0;  // mode 0: quad, 1: paired, 2: all
  int f0_tail = 0;  // merge generation of the CTA's last sequence (the threads that arrive)
  for (int i = 0; i < n; ++i) {
    const int s = i % p.nstage;
    const int r = rw, h = hw, tj = tjw, nt = ntw, gt = a + i;
    if (++tjw == ntw) {
      tjw = 0;
      if (++hw == p.Hkv) {
        hw = 0;
        do {
          ++rw;
        } while (rw < p.num_seqs && tstart[rw + 1] == tstart[rw]);
      }
      if (rw < p.num_seqs) ntw = tstart[rw + 1] - tstart[rw];
    }
    const bool begin = (i == 0) || (tj == 0);
    const bool end = (i == n - 1) || (tj == nt - 1);
    const bool whole = gt - tj >= a && gt - tj + nt <= b;
    bool have = false;
    if (begin) {
      if (!wait_tile(sm, s, (i / p.nstage) & 1, gt)) {
        if (lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
        break;
      }
      if (i == 0 && ctid == 0) trace(T_FIRST_TILE);
      have = true;
      const int qs = seg & 1;
      ++seg;
      const int32_t *qh = sm.misc() + M_QHDR + 8 * qs;
      qlen = qh[2];
      row0 = qh[3];
      L = qh[4];
      mt = qlen;
      paired = mt <= 4;
      // FP8 with one query token: four groups of two warps take every fourth tile, each
      // warp a 64-token half (eight independent accumulator chains per step).  (All eight
      // warps on every tile, 16 tokens each, holds a stage for less time but leaves each
      // warp too little work between its waits: 128K 91.8 against 63.6 us.)
      quad = KVT == PA_KV_FP8_E4M3 && mt == 1;
      if (quad) {
        mode = 0;
        ts = 2;
        active = true;
        mtile = 0;
        sub = warp & 1;
        slice = warp;  // (group, half) = (warp >> 1, warp & 1)
        nsl = 8;
      } else if (paired) {
        mode = 1;
        const int wl = warp & 3;
        ts = 4 / mt;
        active = wl < mt * ts;
        mtile = wl % mt;
        sub = wl / mt;
        slice = (warp >> 2) * ts + sub;
        nsl = 2 * ts;
      } else {
        mode = 2;
        ts = 1;
        active = warp < mt;
        mtile = warp % mt;
        sub = slice = 0;
        nsl = 1;
      }
      cut = L - qlen + mtile + 1;
      if (active) {
        load_q<KVT>(p, sm.qslot(qs) + mtile * kQRowBytes, g, t, f);
        reset_state(f);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.qempty(qs));
    }
    const bool owner = mode == 0 ? (i & 3) == (warp >> 1) : mode == 1 ? (i & 1) == (warp >> 2) : true;
    if (owner) {
      if (!have && !wait_tile(sm, s, (i / p.nstage) & 1, gt)) {
        if (lane == 0) raise_flag(p, sm, PA_DEV_TIMEOUT);
        break;
      }
    }
    if (owner && active) {
      const StageMeta *meta = sm.meta(s);
      const bool masked = (meta->flags & F_MASK) != 0;
      const int tps = kTile / ts;
      const uint32_t st = sm.stage(s);
      if (KVT == PA_KV_FP8_E4M3 && quad) {
        const int tb = sub * 64;
        int pos0[4] = {0, 0, 0, 0};
        if (masked) {
#pragma unroll
          for (int hf = 0; hf < 4; ++hf) {
            const int tk = tb + 16 * hf;
            const int pp = meta->page_pos[tk >> p.ps_shift];
            pos0[hf] = pp < 0 ? -1 : pp + (tk & (p.ps - 1)) + 2 * t;
          }
        }
        chunk_fp8<SM, 8>(p, st, tb, masked, pos0, cut, L, g, t, f);
      } else {
        for (int tb = sub * tps; tb < (sub + 1) * tps; tb += 32) {
          int pos0[2] = {0, 0};
          if (masked) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int tk = tb + 16 * hf;
              const int pp = meta->page_pos[tk >> p.ps_shift];
              pos0[hf] = pp < 0 ? -1 : pp + (tk & (p.ps - 1)) + 2 * t;
            }
          }
          if (KVT == PA_KV_FP8_E4M3)
            chunk_fp8<SM, 4>(p, st, tb, masked, pos0, cut, L, g, t, f);
          else
            chunk_bf16(p, st, tb, masked, pos0, cut, meta->page_pos, L, zero_line(sm), g, t, lane, f);
        }
      }
    }
    if (begin || owner) {
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(sm.empty(s), begin ? 1u : (mode == 0 ? 4u : mode == 1 ? 2u : 1u));
    }

    if (!end) continue;
    if (i == n - 1 && ctid == 0) trace(T_LAST_TILE);  // warp 0 is through the range

    // ---- end of this CTA's part of sequence (r, h): merge the token slices -----------
    // The merge generation of a split sequence, read by the threads that may count this
    // CTA's partial, while the slices merge.  No arrival of this call can have bumped it:
    // that takes every CTA of the sequence, this one included.
    int f0 = 0;
    if (!whole && lane == 0 && active && slice == 0)
      f0 = *reinterpret_cast<volatile int32_t *>(p.flags + r * p.Hkv + h);
    if (SM == PA_SCALE_PER_TOKEN && active) unfold_rows(f);
    const int gs = tstart[r] * p.Hkv + h * nt;
    int c_first = blockIdx.x, nc = 1;
    if (!whole) seq_ctas(p, tstart, r, h, gs, gs + nt, c_first, nc);
    const int slot = slot_of(sm.misc()[M_VCTA], c_first);
    const bool is_head = i < n - 1;
    // At the CTA's last sequence end no tile is in flight any more: every warp puts its
    // state into stage memory and all consumer threads merge the slices element by element,
    // in one step.  Mid-stream ends, and two slices (one round), pair slices through the
    // exchange buffer.
    const bool in_stage = kSlotMerge && !is_head && nsl > 2 && nsl * mt <= kMaxSlots &&
                          p.nstage * p.stage_bytes >= kMaxSlots * kSlotBytes;
    if (in_stage) {
      cons_sync(p, sm, cphase);  // every warp is done with its tiles
      if (active) put_slot(sm.stage(0) + (slice * mt + mtile) * kSlotBytes, f, lane);
      cons_sync(p, sm, cphase);
      merge_slots<KVT>(p, sm.stage(0), nsl, mt, whole, row0, h * kG, slot, ctid);
      if (whole) continue;
    } else {
      // Rounds of pairs through the exchange buffer: the top mv slices (as many as its
      // xslots slots hold, all m-tiles each) merge into the mv below them.
      for (int cnt = nsl; cnt > 1;) {
        const int mv = min(cnt >> 1, p.xslots / mt), lo = cnt - mv;
        if (active && slice >= lo && slice < cnt) put_state(sm, (slice - lo) * mt + mtile, f, lane);
        cons_sync(p, sm, cphase);
        if (active && slice >= lo - mv && slice < lo)
          merge_state(sm, (slice - lo + mv) * mt + mtile, f, lane);
        cons_sync(p, sm, cphase);
        cnt = lo;
      }
      const bool writer = active && slice == 0;
      if (whole) {
        if (writer) write_final<KVT>(p, f, row0 + mtile, h * kG, g, t);
        continue;
      }
      // A split sequence: store this CTA's partial.
      if (writer) write_partial(p, f, slot, mtile, g, t, lane);
    }
    if (i == n - 1 && ctid == 0) trace(T_STORED);
    // The partial is stored.  If the sequence ends before the CTA's last tile it is the one
    // the CTA started in the middle of: it is counted at once (the other warps stream on).
    // The sequence the CTA leaves unfinished is counted after the last tile.
    if (ctid == 0) {
      int32_t *rec = sm.misc() + (is_head ? M_HEAD : M_TAIL);
      rec[0] = r;
      rec[1] = h;
      rec[2] = row0;
      rec[3] = qlen;
      rec[4] = c_first;
      rec[5] = nc;
      sm.misc()[M_F0 + (is_head ? 0 : 1)] = f0;
    }
    if (is_head) {
      has_head = true;
      if (active && slice == 0) {
        __threadfence();
        if (lane == 0) {
          const int w = atomicAdd(&sm.misc()[M_WCNT], 1);
          if (w == mt - 1) {
            sm.misc()[M_WCNT] = 0;
            arrive_split(p, sm, r * p.Hkv + h, nc, f0, 0);
          }
        }
      }
    } else {
      has_tail = true;
      f0_tail = f0;
    }
  }

  if (!(has_head || has_tail)) return;
  if (has_tail) {
    // every consumer thread's partial stores are ordered before the barrier; the one
    // thread that counts the partial fences them for the whole CTA
    cons_sync(p, sm, cphase);
    if (ctid == 0) {
      const int32_t *rec = sm.misc() + M_TAIL;
      __threadfence();
      arrive_split(p, sm, rec[0] * p.Hkv + rec[1], rec[5], f0_tail, 1);
    }
  }
  cons_sync(p, sm, cphase);
  if (ctid == 0) {
    trace(T_ARRIVED);
    trace_value(T_LAST, sm.misc()[M_LAST] | (sm.misc()[M_LAST + 1] << 1));
  }
#pragma unroll 1
  for (int k = 0; k < 2; ++k) {
    const bool mine_k = k == 0 ? has_head : has_tail;
    if (!mine_k) continue;
    const int32_t *rec = sm.misc() + (k == 0 ? M_HEAD : M_TAIL);
    const int hh = rec[1];
    if (kShareMerge && p.coresident && rec[5] * rec[3] >= kShareMin) {
      // every CTA of the sequence takes a share of its merge once all have arrived
      if (!sm.misc()[M_LAST + k]) {
        if (ctid == 0) {
          const int seq = rec[0] * p.Hkv + hh, f0 = sm.misc()[M_F0 + k];
          if (!wait_flag(p.flags + seq, f0)) raise_flag(p, sm, PA_DEV_TIMEOUT);
          __threadfence();
        }
        cons_sync(p, sm, cphase);
      }
      if (ctid == 0) trace(T_MERGE);
      merge_share<KVT>(p, hh, rec[2], rec[3], rec[4], rec[5], sm.misc()[M_VCTA] - rec[4], ctid);
      if (ctid == 0) trace(T_MERGED);
    } else if (sm.misc()[M_LAST + k]) {
      // a small merge, or CTAs of one sequence in different waves: the last to arrive merges
      // alone (the others exit, and the next launch's CTAs take their SMs meanwhile)
      __threadfence();
      if (ctid == 0) trace(T_MERGE);
      merge_partials<KVT>(p, hh, rec[2], rec[3], rec[4], rec[5], ctid);
      if (ctid == 0) trace(T_MERGED);
    }
  }
}

template <int KVT, int SM, bool DUMP>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  const Smem sm = Smem::make(smem_raw + ((1024u - mis) & 1023u), p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), kNCW);
    }
    mbar_init(sm.qempty(0), kNCW);
    mbar_init(sm.qempty(1), kNCW);
    mbar_init(sm.consbar(), kNCW);
    sm.misc()[M_ABORT] = 0;
    sm.misc()[M_LAST] = 0;
    sm.misc()[M_LAST + 1] = 0;
    sm.misc()[M_WCNT] = 0;
    for (int k = 0; k < 4; ++k) sm.misc()[M_ZERO + k] = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 0) trace(T_ENTRY);
  pdl_launch_dependents();
  const uint32_t fl = scan_tiles(p, sm.tstart(), sm.misc() + M_WSUM);
  if (threadIdx.x == 0) {
    trace(T_PROLOGUE);
    trace_value(T_A, (unsigned)sm.misc()[M_WSUM]);
    trace_value(T_B, (unsigned)sm.misc()[M_WSUM + 1]);
  }
  const uint32_t report = blockIdx.x == 0 ? fl : 0u;
  if (warp >= kNCW) {
    regs_dec<kProdRegs>();
    if (warp != kNCW) return;  // the rest of the producer warpgroup only gives registers
    const int a = sm.misc()[M_WSUM], b = sm.misc()[M_WSUM + 1];
    // The producer reads index inputs before the wait, q and the caches after it.
    if (a < b) run_producer<KVT, SM>(p, sm, a, b, report);
    else {
      pdl_wait();
      if (report) atomicOr(p.status, report);
    }
    return;
  }
  regs_inc<kConsRegs>();
  const int a = sm.misc()[M_WSUM], b = sm.misc()[M_WSUM + 1];
  pdl_wait();  // consumers write outputs and the workspace
  if (threadIdx.x == 0) trace(T_CONSUMER);
  if (report) atomicOr(p.status, report);
  run_consumer<KVT, SM, DUMP>(p, sm, a, b, warp, lane);
  if (threadIdx.x == 0) trace_close();
}

// (request, query token, cutoff) of every row, through request_info -- the same map
// the decode kernel uses.
__global__ void row_map_kernel(const __grid_constant__ KParams p, int32_t *row_map) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= p.num_seqs) return;
  uint32_t fl = 0;
  const ReqInfo ri = request_info(p, r, fl);
  for (int tok = 0; tok < ri.qlen; ++tok) {
    const int row = ri.row0 + tok;
    row_map[3 * row] = r;
    row_map[3 * row + 1] = tok;
    row_map[3 * row + 2] = ri.L - ri.qlen + tok + 1;
  }
  if (fl) atomicOr(p.status, fl);
}

}  // namespace pa
