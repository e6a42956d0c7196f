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
// A CTA takes one row at a time and moves on to the next; it has nine
// warps.
//
//   stream  eight warps each read one eighth of the row (a segment) once,
//           each lane keeping its candidates in its own list in shared
//           memory (no warp-wide step to place them).
//           A streaming warp feeds itself: one lane keeps three 2 KB bulk
//           copies of its segment in flight into a ring in shared memory,
//           running on into the warp's segment of the next row, so the
//           stream never waits out a memory latency at a row boundary.
//           A token is kept only when its logit reaches the row's bound
//           L: a value that at least k logits of the row reach, so that
//           nothing below it can be in the top-k.  The eight warps raise L
//           together.  Every kept logit is counted in a histogram of the
//           row that the CTA shares (1/8-binade bins for positive logits,
//           32 coarse bins below zero), and L is the lower edge of
//           the highest bin at and above which k logits have been counted;
//           a warp that finds a better L publishes it for the others.
//           After the first few thousand tokens L sits just below the
//           row's k-th best logit and most steps of 512 tokens keep
//           nothing.  A buffer that fills (L held low by ties or by a
//           narrow spread of logits) is first cleared of entries below L,
//           then cut to its exact top-k; from then on the warp keeps only
//           logits above the k-th best it holds (later tokens have higher
//           ids, so an equal logit ranks below it).
//   merge   the ninth warp concatenates the eight segment lists, cuts them
//           to the row's exact top-k, sorts it into token order and writes
//           the list and (m, Z), while the streaming warps go on to
//           the next row.  Two sets of lists alternate between consecutive
//           rows; named barriers hand a set from the streaming warps to the
//           merging warp and back.
//
// Nothing is dropped that could be in the top-k: an entry leaves a buffer
// only when it is below L or when k entries held rank above it.
//
// Keys are order-preserving unsigned integers of the logit bits (16-bit
// for bf16, 32-bit for fp32), 0 for NaN; -0 counts as +0, so equal logits
// have equal keys.  An exact cut finds the k-th largest key K* by
// narrowing histograms, keeps the keys above K*, and of the entries equal
// to K* those with the lowest ids, up to k in all (found the same way, on
// the ids).
#pragma once

#include "sv_rowpass.cuh"

namespace sv {

constexpr int kTkWarps = 8;                       // streaming warps, one segment of the row each
constexpr int kTkThreads = (kTkWarps + 1) * 32;   // and the merging warp
constexpr int kTkCtasPerSm = 2;                   // resident CTAs per SM (launch bounds)
constexpr int kTkEpl = 16;                        // logits per lane per step
constexpr int kTkStep = 32 * kTkEpl;              // tokens per warp step
constexpr int kTkCapLane = kTkEpl + (SV_MAX_TOPK + 31) / 32;  // a lane's list: a whole
                                                  // step fits after an exact cut
constexpr int kTkCap = 32 * kTkCapLane;           // candidates a streaming warp holds
constexpr int kTkStageBytes = 2048;               // one bulk copy
constexpr int kTkStages = 3;                      // bulk copies in flight per streaming warp
constexpr int kTkSegAlign = 64;                   // segment starts: multiples of 64 tokens
constexpr int kTkNegBins = 32;                    // row histogram: negative logits, coarse
constexpr int kTkBins = kTkNegBins + 2048;        // and the rest in 1/8-binade bins
// named barriers: + the set's parity, lists ready for the merge / set free
// again; and the streaming warps among themselves
constexpr uint32_t kTkBarFull = 1, kTkBarFree = 3, kTkBarStream = 5;

struct TopkPass {
  int n_req, K, V, es, max_topk;
  int seg_len;               // tokens per segment (multiple of kTkSegAlign); 8 segments cover V
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

// Shared memory of one CTA (about 110 KB: two CTAs per SM).
struct TopkShared {
  unsigned char ring[kTkWarps][kTkStages][kTkStageBytes];  // bulk-copy rings
  uint64_t ring_bar[kTkWarps][kTkStages];
  unsigned key[kTkWarps][kTkCap];        // streaming buffers
  int id[kTkWarps][kTkCap];
  unsigned cut_hist[kTkWarps + 1][256];  // scratch of each warp's exact cuts
  unsigned row_hist[kTkBins];            // the row histogram
  unsigned list_key[2][kTkWarps * SV_MAX_TOPK];  // per set: the segments' lists
  int list_id[2][kTkWarps * SV_MAX_TOPK];
  int list_cnt[2][kTkWarps];
  unsigned bad[2];                       // per set: NaN or +inf seen in the row
  unsigned top;                          // highest histogram bin with a count
  unsigned count;                        // logits counted
  unsigned row_lk;                       // the best bound found for the row (a key)
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
__device__ __forceinline__ unsigned tk_key_of(float v, int es) {
  return es == 2 ? tk_key16(__float_as_uint(v) >> 16) : tk_key32(__float_as_uint(v));
}
// Histogram bin of a key.  The bins that set L are those of the row's top
// logits, which are positive in practice: a positive logit (or zero) gets
// one of 2048 bins of 1/8 binade (its exponent and top three mantissa
// bits); the negative logits share 32 coarse bins.  Monotone in the key.
__device__ __forceinline__ unsigned tk_bin(unsigned key, int es) {
  if (es == 2) return key < 0x8000u ? key >> 10 : kTkNegBins + ((key - 0x8000u) >> 4);
  return key < 0x80000000u ? key >> 26 : kTkNegBins + ((key - 0x80000000u) >> 20);
}
// the lowest key of bin b
__device__ __forceinline__ unsigned tk_bin_edge(unsigned b, int es) {
  if (es == 2) return b < kTkNegBins ? b << 10 : 0x8000u + ((b - kTkNegBins) << 4);
  return b < kTkNegBins ? b << 26 : 0x80000000u + ((b - kTkNegBins) << 20);
}
// the largest float below v (v > -inf, not NaN)
__device__ __forceinline__ float tk_below(float v) {
  const unsigned u = __float_as_uint(v);
  if (v > 0.f) return __uint_as_float(u - 1u);
  if (v == 0.f) return __uint_as_float(0x80000001u);
  return __uint_as_float(u + 1u);
}
// NaN-propagating maximum
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ---------------------------------------------------------------- lists
//
// A warp's candidates live in per-lane lists: lane l's i-th entry at index
// l + 32 i of the warp's key / id arrays, i < c (the lane's count).  A
// dense list of n entries is the case c = number of indices l + 32 i < n.
// Entries are kept in no particular order: ties at the k-th value are
// resolved by comparing ids.

// lane l's count in a dense list of n entries
__device__ __forceinline__ int tk_dense_count(int n, int lane) {
  return n > lane ? (n - 1 - lane) / 32 + 1 : 0;
}

// Among the entries of the lists (rows = the largest count), the need-th
// largest of the values that vof gives, over the entries it marks: returns
// (that value V, how many marked entries have a value above V); need >= 1
// and at most the number of marked entries.  V by narrowing a window of
// values that holds it: starting from [min, max] of the marked values, a
// 256-bin histogram of the window (bins 2^shift wide, so the window fills
// the bins), walked down from the top bin until the running count reaches
// the rank still wanted, fixes the bin that holds V; the next window is
// that bin.  Lanes that hit the same bin add once (warp-aggregated).
template <class F>
__device__ __forceinline__ uint2 tk_select(F vof, int rows, int c, unsigned need,
                                           unsigned* hist, int lane) {
  unsigned mn = 0xffffffffu, mx = 0u;
  for (int i = 0; i < rows; ++i) {
    bool in = false;
    unsigned v = 0u;
    if (i < c) in = vof(i, v);
    if (in) {
      mn = min(mn, v);
      mx = max(mx, v);
    }
  }
  unsigned base = __reduce_min_sync(0xffffffffu, mn);
  unsigned span = __reduce_max_sync(0xffffffffu, mx) - base;  // the window: [base, base + span]
  unsigned above_all = 0u;
  for (;;) {
    const int shift = span < 256u ? 0 : 24 - __clz(span);  // (span >> shift) < 256
#pragma unroll
    for (int q = 0; q < 8; ++q) hist[lane * 8 + q] = 0u;
    __syncwarp();
    for (int i = 0; i < rows; ++i) {
      bool in = false;
      unsigned v = 0u;
      if (i < c) in = vof(i, v);
      in = in && v >= base && v - base <= span;
      const unsigned bin = in ? (v - base) >> shift : 0u;
      const unsigned m = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned peers = __match_any_sync(m, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<unsigned>(__popc(peers)));
      }
    }
    __syncwarp();
    // lane l holds bins 255 - 8 l .. 248 - 8 l (descending): lane order is
    // bin order from the top
    unsigned h[8], sum = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      h[q] = hist[255 - 8 * lane - q];
      sum += h[q];
    }
    const unsigned incl = warp_incl_scan_u(sum, lane);
    const unsigned owner = __ffs(__ballot_sync(0xffffffffu, incl >= need)) - 1;
    int bin = 0;
    unsigned above = 0u;
    if (lane == static_cast<int>(owner)) {
      unsigned cum = incl - sum;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum + h[q] >= need && cum < need) {
          bin = 255 - 8 * lane - q;
          above = cum;
        }
        cum += h[q];
      }
    }
    bin = __shfl_sync(0xffffffffu, bin, owner);
    above = __shfl_sync(0xffffffffu, above, owner);
    need -= above;
    above_all += above;
    __syncwarp();
    const unsigned lo = base + (static_cast<unsigned>(bin) << shift);
    if (shift == 0) {
      base = lo;
      break;
    }
    span = min((1u << shift) - 1u, span - (static_cast<unsigned>(bin) << shift));
    base = lo;
  }
  return make_uint2(base, above_all);
}

// Cut the lists (lane count c) to their exact top-k, written back dense:
// the keys above K*, the k-th largest key, and of the keys equal to K*
// those with the lowest ids.  Returns (entries kept, K*).  Lists of at most
// k entries in all are only made dense (K* returned as 0, no key).
__device__ __forceinline__ uint2 tk_cut(unsigned* key, int* id, unsigned* hist, int c, int k,
                                     int lane) {
  __syncwarp();
  const int rows = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(c)));
  const unsigned total = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(c));
  const unsigned lt = (1u << lane) - 1u;
  if (total <= static_cast<unsigned>(k)) {
    unsigned written = 0u;
    for (int i = 0; i < rows; ++i) {
      const bool in = i < c;
      const unsigned kk = in ? key[lane + 32 * i] : 0u;
      const int ii = in ? id[lane + 32 * i] : 0;
      const unsigned km = __ballot_sync(0xffffffffu, in);
      __syncwarp();
      if (in) {
        const unsigned p = written + __popc(km & lt);
        key[p] = kk;
        id[p] = ii;
      }
      written += __popc(km);
      __syncwarp();
    }
    return make_uint2(written, 0u);
  }
  const uint2 ks = tk_select(
      [&](int i, unsigned& v) {
        v = key[lane + 32 * i];
        return true;
      },
      rows, c, static_cast<unsigned>(k), hist, lane);
  const unsigned kstar = ks.x;
  const unsigned need = static_cast<unsigned>(k) - ks.y;  // entries equal to K* to keep
  unsigned ties = 0u;
  for (int i = 0; i < c; ++i) ties += key[lane + 32 * i] == kstar ? 1u : 0u;
  ties = __reduce_add_sync(0xffffffffu, ties);
  // the ties kept: ids up to the need-th smallest (ids are distinct)
  unsigned id_max = 0xffffffffu;
  if (ties > need) {
    const uint2 is = tk_select(
        [&](int i, unsigned& v) {
          v = 0xffffffffu - static_cast<unsigned>(id[lane + 32 * i]);
          return key[lane + 32 * i] == kstar;
        },
        rows, c, need, hist, lane);
    id_max = 0xffffffffu - is.x;
  }
  unsigned written = 0u;
  for (int i = 0; i < rows; ++i) {
    const bool in = i < c;
    const unsigned kk = in ? key[lane + 32 * i] : 0u;
    const int ii = in ? id[lane + 32 * i] : 0;
    const bool keep = in && (kk > kstar || (kk == kstar && static_cast<unsigned>(ii) <= id_max));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // row i is read before any of it is overwritten
    if (keep) {
      const unsigned p = written + __popc(km & lt);  // < 32 (i + 1): rows after i are untouched
      key[p] = kk;
      id[p] = ii;
    }
    written += __popc(km);
    __syncwarp();
  }
  return make_uint2(written, kstar);
}

// Drop the lane's entries below key lk (in place); returns the lane's count.
__device__ __forceinline__ int tk_compact(unsigned* key, int* id, int c, unsigned lk, int lane) {
  int n = 0;
  for (int i = 0; i < c; ++i) {
    const unsigned kk = key[lane + 32 * i];
    if (kk >= lk) {
      id[lane + 32 * n] = id[lane + 32 * i];
      key[lane + 32 * n] = kk;
      ++n;
    }
  }
  return n;
}

// A streaming warp's state for the row.  c is the lane's own count; the
// rest is the same in every lane.
struct TkWarp {
  unsigned* key;  // per-lane lists
  int* id;
  unsigned* hist;  // scratch of the exact cut
  int c;
  unsigned hits;   // steps with a candidate, this row
  unsigned lk;     // the row's bound L as a key; 0: none yet
  unsigned thr;    // the k-th best key held at the warp's last exact cut; 0: none
  float fv, eqv;   // the filter: keep logit x when x > fv or x == eqv
};

// The filter from L (keep x >= value(L)) and the warp's own k-th best
// (keep x > value(thr)).  With neither, every non-NaN logit is kept.
__device__ __forceinline__ void tk_filter(TkWarp& w, int es) {
  const unsigned ninf = es == 2 ? 0x7fu : 0x7fffffu;  // the key of -inf
  const float nan = __int_as_float(0x7fc00000);
  w.fv = kNegInf;
  w.eqv = kNegInf;
  if (w.lk > ninf) {
    w.fv = tk_below(tk_value(w.lk, es));
    w.eqv = nan;
  }
  if (w.thr != 0u) {
    const float t = tk_value(w.thr, es);
    w.fv = w.eqv == w.eqv ? t : fmaxf(w.fv, t);
    w.eqv = nan;
  }
}

// The row's shared state: the histogram, its top bin, the logits counted
// and the best bound any warp has found.
struct TkRowState {
  unsigned* hist;
  unsigned* top;
  unsigned* count;
  unsigned* lk;
};

// Raise L.  The bound any warp found is read every time (one word); the
// histogram is scanned on every fourth step with candidates: L is the lower
// edge of the highest bin b with at least k logits counted at or above it.
// Counts only grow and every counted logit is in the row, so the edge is a
// valid bound whenever it is read.  A bound found is published for the
// other warps.  Other warps move the shared words at any time: lane 0 reads
// them once for the warp, so that every lane takes the same path.
__device__ __forceinline__ void tk_refresh(TkWarp& w, const TkRowState& rs, bool scan, int k,
                                           int es, int lane) {
  unsigned n_seen = 0u, top_b = 0u, shared_lk = 0u;
  if (lane == 0) {
    shared_lk = *reinterpret_cast<volatile unsigned*>(rs.lk);
    if (scan) {
      n_seen = *reinterpret_cast<volatile unsigned*>(rs.count);
      top_b = *reinterpret_cast<volatile unsigned*>(rs.top);
    }
  }
  shared_lk = __shfl_sync(0xffffffffu, shared_lk, 0);
  unsigned lk = max(w.lk, shared_lk);
  if (scan) {
    n_seen = __shfl_sync(0xffffffffu, n_seen, 0);
    top_b = __shfl_sync(0xffffffffu, top_b, 0);
    if (n_seen >= static_cast<unsigned>(k)) {
      const int floor_b = static_cast<int>(tk_bin(lk, es));  // no gain at or below the bound's bin
      const volatile unsigned* hist = rs.hist;
      int hi = static_cast<int>(top_b);
      unsigned carry = 0;
      while (hi > floor_b) {
        const int b = hi - lane;
        const unsigned cb = b > floor_b ? hist[b] : 0u;
        const unsigned incl = warp_incl_scan_u(cb, lane) + carry;
        const unsigned hit =
            __ballot_sync(0xffffffffu, b > floor_b && incl >= static_cast<unsigned>(k));
        if (hit) {
          lk = tk_bin_edge(static_cast<unsigned>(hi - (__ffs(hit) - 1)), es);
          if (lane == 0) atomicMax(rs.lk, lk);
          break;
        }
        carry = __shfl_sync(0xffffffffu, incl, 31);
        hi -= 32;
      }
    }
  }
  if (lk != w.lk) {
    w.lk = lk;
    tk_filter(w, es);
  }
}

// Layout of a step: lane l holds kTkEpl logits in G = ES groups of EPG =
// 16 / ES consecutive tokens (16 bytes each); token of (g, l, j) =
// g * 32 EPG + l * EPG + j.  Each group is one 16-byte load per lane, the
// lanes' loads contiguous.
template <int ES>
struct TkStep {
  static constexpr int kEpg = 16 / ES;      // tokens per group per lane
  static constexpr int kG = kTkEpl / kEpg;  // groups per step
  static constexpr int kSpan = 32 * kEpg;   // tokens per group
};

// the bits of logit j of group words v (j warp-divergent): selects, no
// local memory
template <int ES>
__device__ __forceinline__ unsigned tk_bits(const uint4& v, int j) {
  if constexpr (ES == 2) {
    const unsigned a = (j & 2) ? v.y : v.x, b = (j & 2) ? v.w : v.z;
    const unsigned word = (j & 4) ? b : a;
    return (j & 1) ? (word >> 16) : (word & 0xffffu);
  } else {
    const unsigned a = (j & 1) ? v.y : v.x, b = (j & 1) ? v.w : v.z;
    return (j & 2) ? b : a;
  }
}
// the key of a logit that passed the filter (never NaN)
template <int ES>
__device__ __forceinline__ unsigned tk_key_bits(unsigned x) {
  if constexpr (ES == 2) {
    if (x == 0x8000u) x = 0u;
    return (x & 0x8000u) ? (~x & 0xffffu) : (x | 0x8000u);
  } else {
    if (x == 0x80000000u) x = 0u;
    return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
  }
}
// logit j of group words v as a float (j a constant)
template <int ES>
__device__ __forceinline__ float tk_logit(const uint4& v, int j) {
  const unsigned w4[4] = {v.x, v.y, v.z, v.w};
  if constexpr (ES == 2) return (j & 1) ? bf16hi(w4[j >> 1]) : bf16lo(w4[j >> 1]);
  else return __uint_as_float(w4[j]);
}

// The pass bits of one group (bit j: logit j of the lane's group passes).
template <int ES>
__device__ __forceinline__ unsigned tk_group_pass(const TkWarp& w, const uint4& v) {
  constexpr int E = TkStep<ES>::kEpg;
  unsigned pass = 0;
  if (w.eqv == w.eqv) {  // no bound yet: every non-NaN logit
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const float x = tk_logit<ES>(v, j);
      pass |= (x > w.fv || x == w.eqv) ? (1u << j) : 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) pass |= tk_logit<ES>(v, j) > w.fv ? (1u << j) : 0u;
  }
  return pass;
}

// The pass bits of a step, group g in bits g EPG ..; groups where no lane's
// maximum mg[g] passes are skipped.
template <int ES>
__device__ __forceinline__ unsigned tk_step_pass(const TkWarp& w, const uint4 (&raw)[ES],
                                                 const float (&mg)[ES], unsigned valid) {
  using S = TkStep<ES>;
  unsigned pass = 0;
#pragma unroll
  for (int g = 0; g < S::kG; ++g) {
    const bool gh = !(mg[g] <= w.fv) || mg[g] == w.eqv;
    if (__any_sync(0xffffffffu, gh)) pass |= tk_group_pass<ES>(w, raw[g]) << (g * S::kEpg);
  }
  return pass & valid;
}

// Keep the logits of one step (raw[g], the bits of `valid`; the step starts
// at token id0) that pass the filter: each lane appends its own to its list
// and counts them in the row histogram; then L is raised.  A full list is
// first cleared of entries below L, and the warp's lists are cut to their
// exact top-k if that is not enough.
template <int ES>
__device__ __forceinline__ void tk_take(TkWarp& w, const uint4 (&raw)[ES], unsigned valid,
                                        const float (&mg)[ES], int id0, int k,
                                        const TkRowState& rs, int lane) {
  using S = TkStep<ES>;
  unsigned pass = tk_step_pass<ES>(w, raw, mg, valid);
  int cl = __popc(pass);
  if (__any_sync(0xffffffffu, w.c + cl > kTkCapLane)) {
    w.c = tk_compact(w.key, w.id, w.c, w.lk, lane);
    if (__any_sync(0xffffffffu, w.c + cl > kTkCapLane)) {
      // cut to the exact top-k (or, with at most k entries, spread evenly):
      // at most 64 entries then, two per lane, so a whole step fits
      const uint2 r = tk_cut(w.key, w.id, w.hist, w.c, k, lane);
      w.c = tk_dense_count(static_cast<int>(r.x), lane);
      if (r.y != 0u) {
        w.thr = r.y;
        tk_filter(w, ES);
        pass = tk_step_pass<ES>(w, raw, mg, valid);
        cl = __popc(pass);
      }
    }
  }
  if (cl) {
    unsigned mb = 0u;
    while (pass) {
      const int i = __ffs(pass) - 1;
      pass &= pass - 1u;
      const int g = i / S::kEpg, j = i % S::kEpg;
      uint4 v = raw[0];
#pragma unroll
      for (int q = 1; q < S::kG; ++q)
        if (g == q) v = raw[q];
      const unsigned kk = tk_key_bits<ES>(tk_bits<ES>(v, j));
      w.key[lane + 32 * w.c] = kk;
      w.id[lane + 32 * w.c] = id0 + g * S::kSpan + lane * S::kEpg + j;
      ++w.c;
      const unsigned b = tk_bin(kk, ES);
      atomicAdd(rs.hist + b, 1u);
      mb = max(mb, b);
    }
    atomicMax(rs.top, mb);
    atomicAdd(rs.count, static_cast<unsigned>(cl));
  }
  __syncwarp();
  ++w.hits;
  tk_refresh(w, rs, (w.hits & 3u) == 1u, k, ES, lane);
}

// One step from its raw words (group g in raw[g]; logits beyond the segment
// are -inf and left out of `valid`).  The NaN-propagating maxima tell
// whether any logit can pass and, accumulated in mx, whether the row holds
// NaN or +inf.
template <int ES>
__device__ __forceinline__ void tk_step(TkWarp& w, const uint4 (&raw)[ES], unsigned valid,
                                        int id0, int k, const TkRowState& rs, float& mx,
                                        int lane) {
  float mg[ES];
  if constexpr (ES == 2) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const unsigned m2 = bf16x2_max_nan(bf16x2_max_nan(raw[g].x, raw[g].y),
                                         bf16x2_max_nan(raw[g].z, raw[g].w));
      mg[g] = fmax_nan(bf16lo(m2), bf16hi(m2));
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g)
      mg[g] = fmax_nan(fmax_nan(__uint_as_float(raw[g].x), __uint_as_float(raw[g].y)),
                       fmax_nan(__uint_as_float(raw[g].z), __uint_as_float(raw[g].w)));
  }
  float m = mg[0];
#pragma unroll
  for (int g = 1; g < ES; ++g) m = fmax_nan(m, mg[g]);
  mx = fmax_nan(mx, m);
  const bool hit = !(m <= w.fv) || m == w.eqv;
  if (!__any_sync(0xffffffffu, hit)) return;
  tk_take<ES>(w, raw, valid, mg, id0, k, rs, lane);
}

// The logits of a step at and beyond `n` (segment-relative token `e0` of
// the step's first logit) replaced by -inf, which leaves the step's maximum
// to the tokens of the segment; returns the lane's valid bits.
template <int ES>
__device__ __forceinline__ unsigned tk_mask_tail(uint4 (&raw)[ES], int e0, int n, int lane) {
  using S = TkStep<ES>;
  unsigned valid = 0u;
#pragma unroll
  for (int g = 0; g < S::kG; ++g) {
    const int t0 = e0 + g * S::kSpan + lane * S::kEpg;
    unsigned v[4] = {raw[g].x, raw[g].y, raw[g].z, raw[g].w};
#pragma unroll
    for (int j = 0; j < S::kEpg; ++j) {
      if (t0 + j >= n) {
        if constexpr (ES == 2) {
          const int h = j >> 1;
          v[h] = (j & 1) ? ((v[h] & 0x0000ffffu) | 0xff800000u) : ((v[h] & 0xffff0000u) | 0xff80u);
        } else {
          v[j] = 0xff800000u;
        }
      } else {
        valid |= 1u << (g * S::kEpg + j);
      }
    }
    raw[g] = make_uint4(v[0], v[1], v[2], v[3]);
  }
  return valid;
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
  mbar_arrive_expect_tx(&f.bar[slot], bytes);
  bulk_copy_g2s_hint(f.ring + slot * kTkStageBytes, f.src + off, bytes, &f.bar[slot], f.pol);
  ++f.issued;
  if (++f.stage == f.n_stages) {
    f.stage = 0;
    f.row = tk_next_row(a, f.row + G, G, n_rows);
    if (f.row < n_rows) f.src = tk_row_ptr(a, f.row) + f.seg_off;
  }
}

// Sort 64 items (t = lane: (k0, i0); t = lane + 32: (k1, i1)) by id,
// ascending, with a bitonic network.
__device__ __forceinline__ void tk_cas(unsigned& kk, int& ii, int j, bool asc, int lane) {
  const unsigned ko = __shfl_xor_sync(0xffffffffu, kk, j);
  const int io = __shfl_xor_sync(0xffffffffu, ii, j);
  const bool lower = (lane & j) == 0;
  if (lower == asc ? io < ii : io > ii) {
    kk = ko;
    ii = io;
  }
}
__device__ __forceinline__ void tk_sort64(unsigned& k0, int& i0, unsigned& k1, int& i1, int lane) {
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j == 32) {
        if (i1 < i0) {
          const unsigned tk = k0;
          const int ti = i0;
          k0 = k1;
          i0 = i1;
          k1 = tk;
          i1 = ti;
        }
      } else {
        tk_cas(k0, i0, j, (lane & size) == 0, lane);
        tk_cas(k1, i1, j, ((lane + 32) & size) == 0, lane);
      }
    }
  }
}

// The merging warp: the row's exact top-k from the eight segment lists of
// set p, written out in token order with (m, Z).  The lists are first packed
// together in place.
__device__ void tk_merge(const TopkPass& a, TopkShared& sh, int r, int p, int lane) {
  const int R = 2 * a.K + 1;
  const int b = r / R;
  const int k = a.top_k[b];
  unsigned* key = sh.list_key[p];
  int* id = sh.list_id[p];
  int cnt = 0;
  for (int w = 0; w < kTkWarps; ++w) {
    const int n = __shfl_sync(0xffffffffu, lane == 0 ? sh.list_cnt[p][w] : 0, 0);
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      const unsigned kk = i < n ? key[w * SV_MAX_TOPK + i] : 0u;
      const int ii = i < n ? id[w * SV_MAX_TOPK + i] : 0;
      __syncwarp();  // read before any lane writes (the destination is never ahead)
      if (i < n) {
        key[cnt + i] = kk;
        id[cnt + i] = ii;
      }
      __syncwarp();
    }
    cnt += n;
  }
  if (cnt > k)
    cnt = static_cast<int>(
        tk_cut(key, id, sh.cut_hist[kTkWarps], tk_dense_count(cnt, lane), k, lane).x);
  __syncwarp();
  unsigned k0 = lane < cnt ? key[lane] : 0u, k1 = lane + 32 < cnt ? key[lane + 32] : 0u;
  int i0 = lane < cnt ? id[lane] : 0x7fffffff, i1 = lane + 32 < cnt ? id[lane + 32] : 0x7fffffff;
  tk_sort64(k0, i0, k1, i1, lane);
  const bool bad = __shfl_sync(0xffffffffu, lane == 0 ? sh.bad[p] : 0u, 0) != 0u;
  float2* out = a.lists + static_cast<size_t>(r) * a.max_topk;
  const float v0 = lane < cnt ? tk_value(k0, a.es) : kNegInf;
  const float v1 = lane + 32 < cnt ? tk_value(k1, a.es) : kNegInf;
  if (lane < k) out[lane] = make_float2(v0, __int_as_float(lane < cnt ? i0 : -1));
  if (lane + 32 < k) out[lane + 32] = make_float2(v1, __int_as_float(lane + 32 < cnt ? i1 : -1));
  float m = fmaxf(v0, v1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const Scale2 c = scale_for(a.temperature[b]);
  float z = 0.f;
  if (m != kNegInf) {
    if (lane < cnt) z += fast_exp2(scaled_arg(v0, m, c));
    if (lane + 32 < cnt) z += fast_exp2(scaled_arg(v1, m, c));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) {
    a.mz[r] = bad ? make_float2(__int_as_float(0x7fc00000), 0.f) : make_float2(m, z);
    sh.bad[p] = 0u;
  }
  __syncwarp();
}

// the row's shared state cleared (each warp its eighth of the histogram)
__device__ __forceinline__ void tk_clear_row(TopkShared& sh, int warp, int lane) {
  for (int i = warp * (kTkBins / kTkWarps) + lane; i < (warp + 1) * (kTkBins / kTkWarps); i += 32)
    sh.row_hist[i] = 0u;
  if (warp == 0 && lane == 0) {
    sh.top = 0u;
    sh.count = 0u;
    sh.row_lk = 0u;
  }
}

// A streaming warp: its segment of every row the CTA takes.
template <int ES>
__device__ void tk_stream(const TopkPass& a, TopkShared& sh, int warp, int lane) {
  using S = TkStep<ES>;
  const int n_rows = a.n_req * (2 * a.K + 1);
  const int G = static_cast<int>(gridDim.x);
  const int s0 = warp * a.seg_len;
  const int n = max(0, min(a.seg_len, a.V - s0));  // tokens of the segment (0: none)
  TkWarp w;
  w.key = sh.key[warp];
  w.id = sh.id[warp];
  w.hist = sh.cut_hist[warp];
  const TkRowState rs{sh.row_hist, &sh.top, &sh.count, &sh.row_lk};
  tk_clear_row(sh, warp, lane);
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
  __syncwarp();
  named_sync(kTkBarStream, kTkWarps * 32);
  int r = tk_next_row(a, static_cast<int>(blockIdx.x), G, n_rows);
  for (int p = 0; r < n_rows; p ^= 1) {
    const int b = r / (2 * a.K + 1);
    const int k = a.top_k[b];
    w.c = 0;
    w.hits = 0u;
    w.lk = 0u;
    w.thr = 0u;
    tk_filter(w, ES);
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
#pragma unroll
            for (int g = 0; g < ES; ++g)
              raw[g] = *reinterpret_cast<const uint4*>(stage + (q * kTkStep + g * S::kSpan) * ES +
                                                       lane * 16);
            const unsigned valid =
                eb + kTkStep > n ? tk_mask_tail<ES>(raw, eb, n, lane) : 0xffffu;
            tk_step<ES>(w, raw, valid, s0 + eb, k, rs, mx, lane);
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
        uint4 raw[ES];
#pragma unroll
        for (int g = 0; g < ES; ++g) {
          const int t0 = eb + g * S::kSpan + lane * S::kEpg;
          unsigned v[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
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
          raw[g] = make_uint4(v[0], v[1], v[2], v[3]);
        }
        unsigned valid = 0u;  // tokens of the segment
#pragma unroll
        for (int g = 0; g < S::kG; ++g)
#pragma unroll
          for (int j = 0; j < S::kEpg; ++j)
            if (eb + g * S::kSpan + lane * S::kEpg + j < n) valid |= 1u << (g * S::kEpg + j);
        tk_step<ES>(w, raw, valid, s0 + eb, k, rs, mx, lane);
      }
    }
    const bool bad = mx != mx || mx == kPosInf;
    tk_refresh(w, rs, true, k, ES, lane);
    w.c = tk_compact(w.key, w.id, w.c, w.lk, lane);
    int total = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(w.c)));
    if (total > k) {
      total = static_cast<int>(tk_cut(w.key, w.id, w.hist, w.c, k, lane).x);
      w.c = tk_dense_count(total, lane);
    }
    // hand the segment's list over (set p is free once the row two back is merged)
    const unsigned incl = warp_incl_scan_u(static_cast<unsigned>(w.c), lane);
    const int at = static_cast<int>(incl) - w.c;
    __syncwarp();
    named_sync(kTkBarFree + p, kTkThreads);
    for (int i = 0; i < w.c; ++i) {
      sh.list_key[p][warp * SV_MAX_TOPK + at + i] = w.key[lane + 32 * i];
      sh.list_id[p][warp * SV_MAX_TOPK + at + i] = w.id[lane + 32 * i];
    }
    if (lane == 0) {
      sh.list_cnt[p][warp] = total;
      if (bad) sh.bad[p] = 1u;
    }
    named_arrive(kTkBarFull + p, kTkThreads);
    // every streaming warp is done with the row's shared state: clear it
    named_sync(kTkBarStream, kTkWarps * 32);
    tk_clear_row(sh, warp, lane);
    __syncwarp();
    named_sync(kTkBarStream, kTkWarps * 32);
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
  // the merging warp
  const int n_rows = a.n_req * (2 * a.K + 1);
  const int G = static_cast<int>(gridDim.x);
  if (lane < 2) sh.bad[lane] = 0u;
  int r = tk_next_row(a, static_cast<int>(blockIdx.x), G, n_rows);
  int r2 = r < n_rows ? tk_next_row(a, r + G, G, n_rows) : n_rows;
  __syncwarp();
  if (r < n_rows) named_arrive(kTkBarFree + 0, kTkThreads);
  if (r2 < n_rows) named_arrive(kTkBarFree + 1, kTkThreads);
  for (int p = 0; r < n_rows; p ^= 1) {
    __syncwarp();
    named_sync(kTkBarFull + p, kTkThreads);
    tk_merge(a, sh, r, p, lane);
    const int r3 = r2 < n_rows ? tk_next_row(a, r2 + G, G, n_rows) : n_rows;
    if (r3 < n_rows) named_arrive(kTkBarFree + p, kTkThreads);
    r = r2;
    r2 = r3;
  }
}

}  // namespace sv
