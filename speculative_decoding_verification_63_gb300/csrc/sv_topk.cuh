// sv_topk.cuh -- the top-k lists of filtered rows, a pass of its own that
// runs before the persistent kernel.
//
// With top-k filtering, p and q are each restricted to their own k most
// likely tokens before the accept tests and the residual ("LLM speculative
// decoding study notes 02", sec. 5.4: the draft and the target decode with
// the same strategy; the kept set is the k largest logits, ties at the k-th
// value going to the lower token id).  Neither the accept tests nor the
// residual then need the row again: they need the kept (logit, id) pairs
// and the row's (m, Z) over them.  This pass produces exactly that, per
// filtered row.
//
// A CTA takes one row at a time and moves on to the next; it has ten
// warps.
//
//   stream  eight warps each read one eighth of the row (a segment) once.
//           A streaming warp feeds itself: one lane keeps three 2 KB bulk
//           copies of its segment in flight into a ring in shared memory,
//           running on into the warp's segment of the next row, so the
//           stream never waits out a memory latency at a row boundary.
//           A step is 512 tokens, 16 consecutive tokens per lane.  The lane
//           reduces its 16 logits to their maximum; the maximum of each
//           group of 16 f consecutive tokens (f lanes; f = 1 unless the
//           row's groups would not fit in shared memory) goes into the
//           row's map, one order-preserving key per group, and the lane
//           that leads a group keeps the largest key it wrote.  That is all
//           a step does: no threshold to compare against and no branch on
//           the data, so the pass streams at the speed of the copies.
//   merge   two merging warps take turns, one per map: each takes the
//           finished map of every other row while the streaming warps go on
//           to the next (named barriers hand a map over and back), so a
//           merge has the time of two rows.  Let T be the k-th largest group
//           maximum.  The row's top-k lies within k groups: every group
//           whose maximum is above T (fewer than k), and of the groups whose
//           maximum equals T the first ones in token order, as many as are
//           missing to k.  (A kept logit in a group of maximum T equals T;
//           each of the groups of maximum T before its own holds a logit
//           equal to T with a lower id, and each group above T a logit
//           above T: had its group been left out, k logits would rank above
//           it.)  A first bound is the k-th largest of the lanes' keys: they
//           are the maxima of 256 disjoint unions of groups, so at least k
//           groups reach it.  One scan of the map collects the groups at or
//           above it in token order, typically a few dozen, and T and the
//           chosen groups follow from that short list: T by bisection on
//           the key, then one pass that keeps the groups above T and the
//           first ones equal to T.  A row with too many groups at the first
//           bound (ties spread over the row) takes T by bisection over the
//           whole map and the groups from a scan in token order.  When
//           f > 1 the warp re-reads the chosen groups and applies the same
//           argument to their 16-token pieces.  It then reads the last k
//           pieces (at most 16 k logits) into registers and finds their
//           exact top-k: the k-th largest key K* by bisection, every logit
//           above K*, and of those equal to K* the lowest ids.  The kept
//           logits come out in token order, with (m, Z).
//
// Keys are order-preserving unsigned integers of the logit bits (16-bit
// for bf16, 32-bit for fp32), 0 for NaN; -0 counts as +0, so equal logits
// have equal keys.  A row holding NaN or +inf gets an empty list and
// (m, Z) = (NaN, 0).
#pragma once

#include "sv_rowpass.cuh"

namespace sv {

constexpr int kTkWarps = 8;                       // streaming warps, one segment of the row each
constexpr int kTkMergeWarps = 2;                  // merging warps, one per map parity
constexpr int kTkThreads = (kTkWarps + kTkMergeWarps) * 32;
constexpr int kTkBarCount = (kTkWarps + 1) * 32;  // threads on a hand-over barrier: the
                                                  // streaming warps and one merging warp
constexpr int kTkCtasPerSm = 2;                   // resident CTAs per SM (launch bounds)
constexpr int kTkEpl = 16;                        // consecutive logits per lane per step
constexpr int kTkStep = 32 * kTkEpl;              // tokens per warp step
constexpr int kTkStageBytes = 2048;               // one bulk copy
constexpr int kTkStages = 3;                      // bulk copies in flight per streaming warp
constexpr int kTkMaxFold = 16;                    // lanes per group, at most
constexpr int kTkSegAlign = kTkEpl * kTkMaxFold;  // segment starts: multiples of 256 tokens,
                                                  // so no group straddles two segments
constexpr int kTkMapBytes = 26624;                // one map: a 2- or 4-byte key per group
constexpr int kTkSubCap = SV_MAX_TOPK * kTkMaxFold;  // pieces of the chosen groups
constexpr int kTkListCap = kTkSubCap / 2;         // map entries at or above the first bound
// named barriers: + the map's parity, map ready for the merge / map free
constexpr uint32_t kTkBarFull = 1, kTkBarFree = 3;

struct TopkPass {
  int n_req, K, V, es, max_topk;
  int seg_len;               // tokens per segment (multiple of kTkSegAlign); 8 segments cover V
  int fold;                  // f: lanes per group (a power of two <= kTkMaxFold)
  int group_shift;           // log2(16 f): token >> group_shift is the token's group
  int n_groups;              // groups of the row, ceil(V / 16 f); n_groups * es <= kTkMapBytes
  bool bulk;                 // rows start 16-byte aligned, strides and V * es multiples of
                             // 16 bytes: segments stream through bulk copies
  bool has_draft;
  const char* target;
  int64_t t_stride;          // bytes
  const char* draft;
  int64_t d_stride;
  const int* num_drafts;
  const float* temperature;
  const int* top_k;
  float2* lists;             // [B (2K+1)][max_topk] the row's top-k, token order, padded
                             // with (-inf, -1)
  float2* mz;                // [B (2K+1)] (m, Z) over the kept logits; (NaN, 0) for a row
                             // with NaN or +inf
  int* err;                  // workspace error word (SV_DERR_TIMEOUT)
};

// A merging warp's scratch.
struct TkMergeScratch {
  alignas(16) unsigned sub[kTkSubCap];  // the map's entries at or above the first bound
                                        // (keys, then indices), later the keys of the
                                        // chosen groups' pieces
  int pick[SV_MAX_TOPK];                // the chosen groups
  int start[SV_MAX_TOPK];               // first tokens of the final pieces
};

// Shared memory of one CTA (about 113 KB: two CTAs per SM).
struct TopkShared {
  unsigned char ring[kTkWarps][kTkStages][kTkStageBytes];  // bulk-copy rings
  uint64_t ring_bar[kTkWarps][kTkStages];
  alignas(16) unsigned char map[2][kTkMapBytes];  // per parity: group maxima, zero padded
                                                  // to a multiple of 16 bytes
  unsigned lane_key[2][kTkWarps * 32];  // per parity: each lane's largest group key
  TkMergeScratch ms[kTkMergeWarps];
  unsigned bad[2];                      // per parity: NaN or +inf seen in the row
};

// Order-preserving keys.  bf16: x is the 16-bit pattern; fp32: the 32-bit
// pattern.  NaN -> 0; -0 -> the key of +0.
__device__ __forceinline__ unsigned tk_key16(unsigned x) {
  if (x == 0x8000u) x = 0u;
  if ((x & 0x7fffu) > 0x7f80u) return 0u;
  return (x & 0x8000u) ? (~x & 0xffffu) : (x | 0x8000u);
}
__device__ __forceinline__ unsigned tk_key32(unsigned x) {
  if (x == 0x80000000u) x = 0u;
  if ((x & 0x7fffffffu) > 0x7f800000u) return 0u;
  return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}
// the logit of a key (key != 0)
__device__ __forceinline__ float tk_value(unsigned key, int es) {
  if (es == 2) {
    const unsigned h = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
    return __uint_as_float(h << 16);
  }
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}
// NaN-propagating maximum
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ----------------------------------------------------------- the stream

// The maximum of a lane's 16 logits (ES 16-byte words), NaN-propagating.
template <int ES>
__device__ __forceinline__ float tk_piece_max(const uint4 (&raw)[ES]) {
  if constexpr (ES == 2) {
    const unsigned w = bf16x2_max_nan(
        bf16x2_max_nan(bf16x2_max_nan(raw[0].x, raw[0].y), bf16x2_max_nan(raw[0].z, raw[0].w)),
        bf16x2_max_nan(bf16x2_max_nan(raw[1].x, raw[1].y), bf16x2_max_nan(raw[1].z, raw[1].w)));
    return fmax_nan(bf16lo(w), bf16hi(w));
  } else {
    float m[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
      m[g] = fmax_nan(fmax_nan(__uint_as_float(raw[g].x), __uint_as_float(raw[g].y)),
                      fmax_nan(__uint_as_float(raw[g].z), __uint_as_float(raw[g].w)));
    return fmax_nan(fmax_nan(m[0], m[1]), fmax_nan(m[2], m[3]));
  }
}

// One step: the lane's 16 logits raw (first token t = eb + 16 lane of the
// segment, which holds n tokens and starts at token s0).  Folds the lane
// maxima of each group, writes the group's key to the map and keeps the
// lead lane's largest key.  Called by the whole warp.
template <int ES>
__device__ __forceinline__ void tk_step(const TopkPass& a, const uint4 (&raw)[ES], int eb, int n,
                                        int s0, unsigned char* map, unsigned& lkey, float& mx,
                                        int lane) {
  const float m = tk_piece_max<ES>(raw);
  mx = fmax_nan(mx, m);
  unsigned key = ES == 2 ? tk_key16(__float_as_uint(m) >> 16) : tk_key32(__float_as_uint(m));
  for (int o = 1; o < a.fold; o <<= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  const int t = eb + kTkEpl * lane;
  if ((lane & (a.fold - 1)) == 0 && t < n) {
    const int g = (s0 + t) >> a.group_shift;
    if (!SV_CHECK(g < a.n_groups, a.err)) return;
    if constexpr (ES == 2) reinterpret_cast<unsigned short*>(map)[g] = static_cast<unsigned short>(key);
    else reinterpret_cast<unsigned*>(map)[g] = key;
    lkey = max(lkey, key);
  }
}

// The lane's logits at and beyond segment token n replaced by -inf (t: the
// segment token of the lane's first logit), which leaves the maximum to the
// tokens of the segment.
template <int ES>
__device__ __forceinline__ void tk_mask_tail(uint4 (&raw)[ES], int t, int n) {
  constexpr int E = 16 / ES;  // logits per word
#pragma unroll
  for (int g = 0; g < ES; ++g) {
    unsigned v[4] = {raw[g].x, raw[g].y, raw[g].z, raw[g].w};
#pragma unroll
    for (int j = 0; j < E; ++j) {
      if (t + g * E + j >= n) {
        if constexpr (ES == 2) {
          const int h = j >> 1;
          v[h] = (j & 1) ? ((v[h] & 0x0000ffffu) | 0xff800000u) : ((v[h] & 0xffff0000u) | 0xff80u);
        } else {
          v[j] = 0xff800000u;
        }
      }
    }
    raw[g] = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// the row of index r (b, i): target rows 0..nd, then the nd draft rows
__device__ __forceinline__ const char* tk_row_ptr(const TopkPass& a, int r) {
  const int R = 2 * a.K + 1;
  const int b = r / R, rl = r % R;
  const int nd = a.num_drafts ? a.num_drafts[b] : a.K;
  return rl <= nd ? a.target + (static_cast<int64_t>(b) * (a.K + 1) + rl) * a.t_stride
                  : a.draft + (static_cast<int64_t>(b) * a.K + (rl - nd - 1)) * a.d_stride;
}

// the first row at or after r, stepping by `step`, that the pass filters;
// n_rows when there is none
__device__ __forceinline__ int tk_next_row(const TopkPass& a, int r, int step, int n_rows) {
  const int R = 2 * a.K + 1;
  for (; r < n_rows; r += step) {
    const int b = r / R, rl = r % R;
    const int nd = a.num_drafts ? a.num_drafts[b] : a.K;
    const int k = a.top_k ? a.top_k[b] : 0;
    if (chain_kind(nd, a.temperature[b], k, a.K, a.V, a.max_topk, a.has_draft) == KIND_TOPK &&
        rl <= 2 * nd)
      return r;
  }
  return n_rows;
}

// The bulk copies of one streaming warp: stage s of the warp's stream (its
// segment of each of the CTA's rows in turn, 2 KB at a time) goes to ring
// slot s % kTkStages.  Lane 0 issues; `issued` runs kTkStages ahead of the
// stages consumed.
struct TkFeed {
  unsigned char* ring;
  uint64_t* bar;
  uint64_t pol;
  int row, stage;     // the next stage to issue: row index and stage within the row
  const char* src;    // the segment of that row
  int n_stages;       // stages per row (the segment, 2 KB at a time)
  int seg_bytes;      // bytes of the segment
  int64_t seg_off;    // byte offset of the segment within a row
  unsigned issued, consumed;
  int put, take;          // ring slots of the next issue and the next consumption
  unsigned take_phase;    // parity of the next consumption's phase
};

__device__ __forceinline__ void tk_feed_issue(TkFeed& f, const TopkPass& a, int G, int n_rows) {
  if (f.row >= n_rows || f.n_stages == 0) return;
  const int slot = f.put;
  f.put = f.put + 1 == kTkStages ? 0 : f.put + 1;
  const int off = f.stage * kTkStageBytes;
  const uint32_t bytes = static_cast<uint32_t>(min(kTkStageBytes, f.seg_bytes - off));
  fence_proxy_async_shared();  // the slot's earlier reads before the copy's writes
  if (SV_CHECK(bulk_args_ok(f.ring + slot * kTkStageBytes, f.src + off, bytes) &&
                   off + static_cast<int>(bytes) <= f.seg_bytes,
               a.err)) {
    mbar_arrive_expect_tx(&f.bar[slot], bytes);
    bulk_copy_g2s_hint(f.ring + slot * kTkStageBytes, f.src + off, bytes, &f.bar[slot], f.pol);
  } else {
    mbar_arrive(&f.bar[slot]);  // nothing copied: the stage completes empty
  }
  ++f.issued;
  if (++f.stage == f.n_stages) {
    f.stage = 0;
    f.row = tk_next_row(a, f.row + G, G, n_rows);
    if (f.row < n_rows) f.src = tk_row_ptr(a, f.row) + f.seg_off;
  }
}

// A streaming warp: its segment of every row the CTA takes, into the map
// of the row's parity.
template <int ES>
__device__ void tk_stream(const TopkPass& a, TopkShared& sh, int warp, int lane) {
  const int n_rows = a.n_req * (2 * a.K + 1);
  const int G = static_cast<int>(gridDim.x);
  const int s0 = warp * a.seg_len;
  const int n = max(0, min(a.seg_len, a.V - s0));  // tokens of the segment (0: none)
  TkFeed f;
  f.ring = &sh.ring[warp][0][0];
  f.bar = sh.ring_bar[warp];
  f.pol = policy_evict_first();
  f.seg_bytes = n * ES;
  f.seg_off = static_cast<int64_t>(s0) * ES;
  f.n_stages = a.bulk ? (f.seg_bytes + kTkStageBytes - 1) / kTkStageBytes : 0;
  f.row = tk_next_row(a, static_cast<int>(blockIdx.x), G, n_rows);
  f.src = f.row < n_rows ? tk_row_ptr(a, f.row) + f.seg_off : nullptr;
  f.stage = 0;
  f.issued = 0u;
  f.consumed = 0u;
  f.put = 0;
  f.take = 0;
  f.take_phase = 0u;
  if (f.n_stages > 0) {
    if (lane == 0) {
      for (int i = 0; i < kTkStages; ++i) mbar_init(&f.bar[i], 1);
      fence_mbar_init();
      for (int i = 0; i < kTkStages; ++i) tk_feed_issue(f, a, G, n_rows);
    }
    __syncwarp();
  }
  bool timed_out = false;
  int r = tk_next_row(a, static_cast<int>(blockIdx.x), G, n_rows);
  for (int p = 0; r < n_rows; p ^= 1) {
    // the merge is done with this parity's map (the row two back)
    named_sync(kTkBarFree + p, kTkBarCount);
    unsigned char* map = sh.map[p];
    unsigned lkey = 0u;
    float mx = kNegInf;
    if (a.bulk) {
      for (int st = 0; st < f.n_stages; ++st) {
        const int slot = f.take;
        const uint32_t parity = f.take_phase;
        // every lane waits on the copy itself (the wait is what makes the
        // copied bytes visible to it)
        bool ok = timed_out || mbar_wait_bounded(&f.bar[slot], parity, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) record_error(a.err, SV_DERR_TIMEOUT);
          timed_out = true;
        }
        if (!timed_out) {
          const unsigned char* stage = f.ring + slot * kTkStageBytes;
          constexpr int kStageEl = kTkStageBytes / ES;
#pragma unroll
          for (int q = 0; q < kStageEl / kTkStep; ++q) {
            const int eb = st * kStageEl + q * kTkStep;  // segment-relative
            if (eb >= n) break;                          // warp-uniform
            uint4 raw[ES];
            const unsigned char* src = stage + (q * kTkStep + lane * kTkEpl) * ES;
#pragma unroll
            for (int g = 0; g < ES; ++g) raw[g] = *reinterpret_cast<const uint4*>(src + 16 * g);
            if (eb + kTkStep > n) tk_mask_tail<ES>(raw, eb + kTkEpl * lane, n);
            tk_step<ES>(a, raw, eb, n, s0, map, lkey, mx, lane);
          }
        }
        __syncwarp();  // every lane is done with the slot
        ++f.consumed;
        if (++f.take == kTkStages) {
          f.take = 0;
          f.take_phase ^= 1u;
        }
        if (lane == 0 && !timed_out) tk_feed_issue(f, a, G, n_rows);
      }
    } else {
      // rows not fit for bulk copies: the same steps from plain loads
      const char* row = tk_row_ptr(a, r) + static_cast<int64_t>(s0) * ES;
      for (int eb = 0; eb < n; eb += kTkStep) {
        const int t0 = eb + kTkEpl * lane;
        unsigned v[4 * ES];
#pragma unroll
        for (int h = 0; h < 4 * ES; ++h) {
          if constexpr (ES == 2) {
            const int t = t0 + 2 * h;
            const unsigned lo = t < n ? __ldg(reinterpret_cast<const unsigned short*>(row) + t)
                                      : 0xff80u;
            const unsigned hi = t + 1 < n
                ? __ldg(reinterpret_cast<const unsigned short*>(row) + t + 1) : 0xff80u;
            v[h] = lo | (hi << 16);
          } else {
            const int t = t0 + h;
            v[h] = t < n ? __ldg(reinterpret_cast<const unsigned*>(row) + t) : 0xff800000u;
          }
        }
        uint4 raw[ES];
#pragma unroll
        for (int g = 0; g < ES; ++g)
          raw[g] = make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        tk_step<ES>(a, raw, eb, n, s0, map, lkey, mx, lane);
      }
    }
    // hand the map over
    sh.lane_key[p][warp * 32 + lane] = lkey;
    const bool bad = __any_sync(0xffffffffu, mx != mx || mx == kPosInf);
    if (bad && lane == 0) sh.bad[p] = 1u;
    named_arrive(kTkBarFull + p, kTkBarCount);
    r = tk_next_row(a, r + G, G, n_rows);
  }
  // after a timeout, copies may still be in flight into the ring: wait for
  // them (briefly) before the CTA's shared memory is released
  if (lane == 0)
    for (; f.consumed < f.issued; ++f.consumed) {
      mbar_wait_bounded(&f.bar[f.take], f.take_phase, kWaitLimitAfterTimeoutNs);
      if (++f.take == kTkStages) {
        f.take = 0;
        f.take_phase ^= 1u;
      }
    }
  __syncwarp();
}

// ------------------------------------------------------------ the merge

// key e of a 16-byte word of KB-byte keys
template <int KB>
__device__ __forceinline__ unsigned tk_word_key(const uint4& w, int e) {
  if constexpr (KB == 2) {
    const unsigned x = (e >> 1) == 0 ? w.x : (e >> 1) == 1 ? w.y : (e >> 1) == 2 ? w.z : w.w;
    return (e & 1) ? (x >> 16) : (x & 0xffffu);
  } else {
    return e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w;
  }
}

// How many keys of an array of n16 16-byte words of KB-byte keys (zero
// padded) are >= v (v >= 1).
template <int KB>
__device__ __forceinline__ unsigned tk_count_ge(const uint4* m, int n16, unsigned v, int lane) {
  unsigned c = 0u;
  if constexpr (KB == 2) {
    const unsigned v2 = v | (v << 16);
#pragma unroll 4
    for (int i = lane; i < n16; i += 32) {
      const uint4 w = m[i];
      // 0xffff per half at or above v: 16 bits per key counted
      c += __popc(__vcmpgeu2(w.x, v2)) + __popc(__vcmpgeu2(w.y, v2)) +
           __popc(__vcmpgeu2(w.z, v2)) + __popc(__vcmpgeu2(w.w, v2));
    }
    c >>= 4;
  } else {
#pragma unroll 4
    for (int i = lane; i < n16; i += 32) {
      const uint4 w = m[i];
      c += (w.x >= v ? 1u : 0u) + (w.y >= v ? 1u : 0u) + (w.z >= v ? 1u : 0u) +
           (w.w >= v ? 1u : 0u);
    }
  }
  return __reduce_add_sync(0xffffffffu, c);
}

// The largest key T with at least k keys >= T, by bisection from lo (at
// least k keys reach it) and hi > lo (fewer than k reach it; n_hi of
// them).  Returns (T, the number of keys above T).
template <int KB>
__device__ uint2 tk_kth(const uint4* m, int n16, int k, unsigned lo, unsigned hi, unsigned n_hi,
                        int lane) {
  while (hi - lo > 1u) {
    const unsigned mid = lo + ((hi - lo) >> 1);
    const unsigned c = tk_count_ge<KB>(m, n16, mid, lane);
    if (c >= static_cast<unsigned>(k)) {
      lo = mid;
    } else {
      hi = mid;
      n_hi = c;
    }
  }
  return make_uint2(lo, n_hi);
}

// The chosen entries of a key array, in index order: every key above T,
// and of the keys equal to T the first `quota`.  Their indices go to
// out[0 ..]; returns how many (at most cap; the scan stops there).
template <int KB>
__device__ int tk_pick(const uint4* m, int n16, unsigned T, int quota, int* out, int cap,
                       int lane) {
  constexpr int E = 16 / KB;  // keys per word
  int written = 0, eq_seen = 0;
  for (int i0 = 0; i0 < n16 && written < cap; i0 += 32) {
    const int i = i0 + lane;
    unsigned gt = 0u, eq = 0u;
    if (i < n16) {
      const uint4 w = m[i];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned key = tk_word_key<KB>(w, e);
        gt |= (key > T ? 1u : 0u) << e;
        eq |= (key == T ? 1u : 0u) << e;
      }
    }
    // the ties this lane may keep: the first (quota - ties before it)
    const int ne = __popc(eq);
    const int eq_incl = static_cast<int>(warp_incl_scan_u(static_cast<unsigned>(ne), lane));
    const int room = quota - (eq_seen + eq_incl - ne);
    unsigned eq_keep = eq;
    for (int drop = ne - max(0, room); drop > 0; --drop) eq_keep &= ~(1u << (31 - __clz(eq_keep)));
    const unsigned keep = gt | eq_keep;
    const int nk = __popc(keep);
    const int k_incl = static_cast<int>(warp_incl_scan_u(static_cast<unsigned>(nk), lane));
    int at = written + k_incl - nk;
    for (unsigned b = keep; b; b &= b - 1u, ++at)
      if (at < cap) out[at] = i * E + (__ffs(b) - 1);
    written += __shfl_sync(0xffffffffu, k_incl, 31);
    eq_seen += __shfl_sync(0xffffffffu, eq_incl, 31);
  }
  __syncwarp();
  return min(written, cap);
}

// The entries of a key array (n16 16-byte words of KB-byte keys) whose key
// is at least lo, in index order: keys to key[], indices to idx[] (the
// first kTkListCap of them).  Returns how many there are.  Few entries
// reach the bound, so a word is mostly one test; a lane's place in the list
// comes from ballots of the bits of its count (at most 8), no atomics.
template <int KB>
__device__ __forceinline__ int tk_collect(const uint4* m, int n16, unsigned lo, unsigned* key,
                                          int* idx, int lane) {
  constexpr int E = 16 / KB;  // keys per word
  const unsigned lt = (1u << lane) - 1u;
  int total = 0;
#pragma unroll 2
  for (int i0 = 0; i0 < n16; i0 += 32) {
    const int i = i0 + lane;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    unsigned hits = 0u;
    if (i < n16) {
      w = m[i];
#pragma unroll
      for (int e = 0; e < E; ++e) hits |= (tk_word_key<KB>(w, e) >= lo ? 1u : 0u) << e;
    }
    if (__any_sync(0xffffffffu, hits != 0u)) {
      const unsigned c = static_cast<unsigned>(__popc(hits));
      const unsigned b0 = __ballot_sync(0xffffffffu, c & 1u);
      const unsigned b1 = __ballot_sync(0xffffffffu, c & 2u);
      const unsigned b2 = __ballot_sync(0xffffffffu, c & 4u);
      const unsigned b3 = __ballot_sync(0xffffffffu, c & 8u);
      int at = total + __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt) +
               8 * __popc(b3 & lt);
      for (; hits; hits &= hits - 1u, ++at) {
        const int e = __ffs(hits) - 1;
        if (at < kTkListCap) {
          key[at] = tk_word_key<KB>(w, e);
          idx[at] = i * E + e;
        }
      }
      total += __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2) + 8 * __popc(b3);
    }
  }
  __syncwarp();
  return total;
}

// The chosen groups from the list of the map's entries at or above lo
// (keys key[], map indices idx[] ascending, n of them; at least k): with T
// the k-th largest key, every entry above T and of those equal to T the
// first ones, k in all, written to out[] in list order.  hi: above every
// key.  Returns T.
__device__ unsigned tk_pick_list(const unsigned* key, const int* idx, int n, int k, unsigned lo,
                                 unsigned hi, int* out, int lane) {
  unsigned n_hi = 0u;
  while (hi - lo > 1u) {
    const unsigned mid = lo + ((hi - lo) >> 1);
    unsigned c = 0u;
    for (int j = lane; j < n; j += 32) c += key[j] >= mid ? 1u : 0u;
    c = __reduce_add_sync(0xffffffffu, c);
    if (c >= static_cast<unsigned>(k)) {
      lo = mid;
    } else {
      hi = mid;
      n_hi = c;
    }
  }
  const unsigned T = lo;
  const int quota = k - static_cast<int>(n_hi);  // entries equal to T to keep
  const unsigned lt = (1u << lane) - 1u;
  int written = 0, ties = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const unsigned kj = j < n ? key[j] : 0u;
    const bool tie = j < n && kj == T;
    const unsigned bt = __ballot_sync(0xffffffffu, tie);
    const bool keep = (j < n && kj > T) || (tie && ties + __popc(bt & lt) < quota);
    const unsigned bk = __ballot_sync(0xffffffffu, keep);
    if (keep && written + __popc(bk & lt) < k) out[written + __popc(bk & lt)] = idx[j];
    written += __popc(bk);
    ties += __popc(bt);
  }
  __syncwarp();
  return T;
}

// The keys of the 16 logits from token t0 of a row (0 beyond V): vector
// loads when the row is 16-byte aligned and the piece whole.
template <int ES>
__device__ __forceinline__ void tk_piece_keys(const char* row, int t0, int V, bool vec,
                                              unsigned (&kk)[kTkEpl]) {
  if (vec && t0 + kTkEpl <= V) {
    const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<int64_t>(t0) * ES);
#pragma unroll
    for (int g = 0; g < ES; ++g) {
      const uint4 w = __ldg(p + g);
      const unsigned x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if constexpr (ES == 2) {
          kk[8 * g + 2 * h] = tk_key16(x[h] & 0xffffu);
          kk[8 * g + 2 * h + 1] = tk_key16(x[h] >> 16);
        } else {
          kk[4 * g + h] = tk_key32(x[h]);
        }
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kTkEpl; ++j) {
      const int t = t0 + j;
      if constexpr (ES == 2)
        kk[j] = t < V ? tk_key16(__ldg(reinterpret_cast<const unsigned short*>(row) + t)) : 0u;
      else
        kk[j] = t < V ? tk_key32(__ldg(reinterpret_cast<const unsigned*>(row) + t)) : 0u;
    }
  }
}

// The exact top-k of the n (<= 64) 16-token pieces starting at tokens
// start[0 ..] (ascending), written in token order to out with (m, Z).  lo:
// a key that at least k of the pieces' logits reach.
template <int ES>
__device__ void tk_final(const TopkPass& a, const char* row, const int* start, int n, int k,
                         unsigned lo, float temperature, float2* out, float2* mz, int lane) {
  unsigned kk[2][kTkEpl];
  int t0[2];
  unsigned top = 0u;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    t0[s] = i < n ? start[i] : -1;
    if (t0[s] >= 0 && !SV_CHECK(t0[s] < a.V && (t0[s] & (kTkEpl - 1)) == 0, a.err)) t0[s] = -1;
    if (t0[s] >= 0) {
      tk_piece_keys<ES>(row, t0[s], a.V, a.bulk, kk[s]);
    } else {
#pragma unroll
      for (int j = 0; j < kTkEpl; ++j) kk[s][j] = 0u;
    }
#pragma unroll
    for (int j = 0; j < kTkEpl; ++j) top = max(top, kk[s][j]);
  }
  const unsigned hi0 = __reduce_max_sync(0xffffffffu, top) + 1u;
  lo = max(lo, 1u);  // tokens beyond V (key 0) never count
  if (lo >= hi0) lo = hi0 - 1u;
  // K* = the k-th largest key, by bisection; n_gt keys above it
  unsigned hi = hi0, n_gt = 0u;
  while (hi - lo > 1u) {
    const unsigned mid = lo + ((hi - lo) >> 1);
    unsigned c = 0u;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int j = 0; j < kTkEpl; ++j) c += kk[s][j] >= mid ? 1u : 0u;
    c = __reduce_add_sync(0xffffffffu, c);
    if (c >= static_cast<unsigned>(k)) {
      lo = mid;
    } else {
      hi = mid;
      n_gt = c;
    }
  }
  const unsigned kstar = lo;
  const int quota = k - static_cast<int>(n_gt);  // logits equal to K* to keep
  // keep masks per piece; ties counted in token order (pieces lane, then
  // lane + 32)
  unsigned gt[2], eq[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    gt[s] = 0u;
    eq[s] = 0u;
#pragma unroll
    for (int j = 0; j < kTkEpl; ++j) {
      gt[s] |= (kk[s][j] > kstar && kstar >= 1u ? 1u : 0u) << j;
      eq[s] |= (kk[s][j] == kstar && kstar >= 1u ? 1u : 0u) << j;
    }
  }
  int tie_base = 0, out_base = 0;
  unsigned keep[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int ne = __popc(eq[s]);
    const int eq_incl = static_cast<int>(warp_incl_scan_u(static_cast<unsigned>(ne), lane));
    const int room = quota - (tie_base + eq_incl - ne);
    unsigned ek = eq[s];
    for (int drop = ne - max(0, room); drop > 0; --drop) ek &= ~(1u << (31 - __clz(ek)));
    keep[s] = gt[s] | ek;
    tie_base += __shfl_sync(0xffffffffu, eq_incl, 31);
  }
  // (m, Z): the largest key is kept whenever anything is
  const float m = hi0 > 1u ? tk_value(hi0 - 1u, ES) : kNegInf;
  const Scale2 c = scale_for(temperature);
  float z = 0.f;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int nk = __popc(keep[s]);
    const int k_incl = static_cast<int>(warp_incl_scan_u(static_cast<unsigned>(nk), lane));
    const int at0 = out_base + k_incl - nk;
#pragma unroll
    for (int j = 0; j < kTkEpl; ++j) {
      if ((keep[s] >> j) & 1u) {
        const int at = at0 + __popc(keep[s] & ((1u << j) - 1u));
        const float v = tk_value(kk[s][j], ES);
        if (at < k) out[at] = make_float2(v, __int_as_float(t0[s] + j));
        if (m != kNegInf) z += fast_exp2(scaled_arg(v, m, c));
      }
    }
    out_base += __shfl_sync(0xffffffffu, k_incl, 31);
  }
  for (int i = out_base + lane; i < k; i += 32) out[i] = make_float2(kNegInf, __int_as_float(-1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) *mz = make_float2(m, z);
  __syncwarp();
}

// The merging warp, row r from the map of parity p.  The map is released
// (release: another row will use it) as soon as the groups are chosen.
template <int ES>
__device__ void tk_merge(const TopkPass& a, TopkShared& sh, TkMergeScratch& ms, int r, int p,
                         bool release, int lane) {
  const int R = 2 * a.K + 1;
  const int b = r / R;
  const int k = a.top_k[b];
  const int f = a.fold;
  const bool bad = __shfl_sync(0xffffffffu, lane == 0 ? sh.bad[p] : 0u, 0) != 0u;
  int n_pick = 0;
  unsigned T = 1u;
  if (!bad) {
    if (a.n_groups <= k) {
      n_pick = a.n_groups;
      for (int i = lane; i < n_pick; i += 32) ms.pick[i] = i;
    } else {
      // a first bound from the lanes' keys: their k-th largest
      unsigned lk[8], mn = 0xffffffffu, mxk = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        lk[q] = sh.lane_key[p][8 * lane + q];
        mn = min(mn, lk[q]);
        mxk = max(mxk, lk[q]);
      }
      unsigned lo = __reduce_min_sync(0xffffffffu, mn);
      unsigned hi = __reduce_max_sync(0xffffffffu, mxk) + 1u;
      const unsigned top1 = hi;
      while (hi - lo > 1u) {
        const unsigned mid = lo + ((hi - lo) >> 1);
        unsigned c = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) c += lk[q] >= mid ? 1u : 0u;
        c = __reduce_add_sync(0xffffffffu, c);
        if (c >= static_cast<unsigned>(k)) lo = mid;
        else hi = mid;
      }
      // the map's entries at or above that bound: T and the chosen groups
      // from them, unless there are too many (ties spread over the row):
      // then by bisection over the whole map and a scan in token order
      const uint4* map = reinterpret_cast<const uint4*>(sh.map[p]);
      const int n16 = (a.n_groups * ES + 15) / 16;
      unsigned* list_key = ms.sub;
      int* list_idx = reinterpret_cast<int*>(ms.sub + kTkListCap);
      const int n_c = lo >= 1u ? tk_collect<ES>(map, n16, lo, list_key, list_idx, lane) : 0;
      if (lo >= 1u && n_c <= kTkListCap) {
        T = tk_pick_list(list_key, list_idx, n_c, k, lo, top1, ms.pick, lane);
        n_pick = k;
      } else {
        const uint2 t = tk_kth<ES>(map, n16, k, lo, top1, 0u, lane);
        T = t.x;
        n_pick = tk_pick<ES>(map, n16, t.x, k - static_cast<int>(t.y), ms.pick, k, lane);
      }
    }
  }
  __syncwarp();
  if (lane == 0) sh.bad[p] = 0u;
  if (release) named_arrive(kTkBarFree + p, kTkBarCount);

  const char* row = tk_row_ptr(a, r);
  float2* out = a.lists + static_cast<size_t>(r) * a.max_topk;
  if (bad) {
    for (int i = lane; i < k; i += 32) out[i] = make_float2(kNegInf, __int_as_float(-1));
    if (lane == 0) a.mz[r] = make_float2(__int_as_float(0x7fc00000), 0.f);
    __syncwarp();
    return;
  }
  int n_start = n_pick;
  if (f == 1) {
    for (int i = lane; i < n_pick; i += 32) ms.start[i] = ms.pick[i] * kTkEpl;
  } else {
    // the chosen groups' 16-token pieces, in token order, and their keys
    const int n_sub = n_pick * f;
    const int n_sub4 = (n_sub + 3) & ~3;
    unsigned top = 0u;
    for (int s = lane; s < n_sub4; s += 32) {
      unsigned key = 0u;
      if (s < n_sub) {
        unsigned kk[kTkEpl];
        tk_piece_keys<ES>(row, (ms.pick[s / f] * f + s % f) * kTkEpl, a.V, a.bulk, kk);
#pragma unroll
        for (int j = 0; j < kTkEpl; ++j) key = max(key, kk[j]);
      }
      ms.sub[s] = key;
      top = max(top, key);
    }
    __syncwarp();
    if (n_sub <= k) {
      n_start = n_sub;
      for (int s = lane; s < n_sub; s += 32) ms.start[s] = s;
    } else {
      const uint4* sub = reinterpret_cast<const uint4*>(ms.sub);
      const unsigned top1 = __reduce_max_sync(0xffffffffu, top) + 1u;
      const uint2 t = tk_kth<4>(sub, n_sub4 / 4, k, max(T, 1u), top1, 0u, lane);
      T = t.x;
      n_start = tk_pick<4>(sub, n_sub4 / 4, t.x, k - static_cast<int>(t.y), ms.start, k, lane);
    }
    for (int i = lane; i < n_start; i += 32) {
      const int s = ms.start[i];
      ms.start[i] = (ms.pick[s / f] * f + s % f) * kTkEpl;
    }
  }
  __syncwarp();
  tk_final<ES>(a, row, ms.start, n_start, k, T, a.temperature[b], out, a.mz + r, lane);
}

__global__ void __launch_bounds__(kTkThreads, kTkCtasPerSm) topk_kernel(const TopkPass a) {
  extern __shared__ __align__(128) unsigned char tk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(tk_smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_launch_dependents();
  if (warp < kTkWarps) {
    if (a.es == 2) tk_stream<2>(a, sh, warp, lane);
    else tk_stream<4>(a, sh, warp, lane);
    return;
  }
  // merging warp m takes the CTA's rows of parity m (every other row, from
  // the m-th).  The padding of its map (never written by the stream) reads
  // as key 0.
  const int m = warp - kTkWarps;
  const int n_rows = a.n_req * (2 * a.K + 1);
  const int G = static_cast<int>(gridDim.x);
  const int used = a.n_groups * a.es;
  for (int i = used + lane; i < ((used + 15) & ~15); i += 32) sh.map[m][i] = 0u;
  if (lane == 0) sh.bad[m] = 0u;
  auto next = [&](int x) { return x < n_rows ? tk_next_row(a, x + G, G, n_rows) : n_rows; };
  int r = tk_next_row(a, static_cast<int>(blockIdx.x), G, n_rows);
  if (m == 1) r = next(r);
  __syncwarp();
  if (r < n_rows) named_arrive(kTkBarFree + m, kTkBarCount);
  while (r < n_rows) {
    __syncwarp();
    named_sync(kTkBarFull + m, kTkBarCount);
    const int rn = next(next(r));
    if (a.es == 2) tk_merge<2>(a, sh, sh.ms[m], r, m, rn < n_rows, lane);
    else tk_merge<4>(a, sh, sh.ms[m], r, m, rn < n_rows, lane);
    r = rn;
  }
}

}  // namespace sv
