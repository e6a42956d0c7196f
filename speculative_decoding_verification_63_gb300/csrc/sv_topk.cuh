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
//           keeping candidates in their own shared buffer, in token order.
//           A streaming warp feeds itself: one lane keeps three 2 KB bulk
//           copies of its segment in flight into a ring in shared memory,
//           running on into the warp's segment of the next row, so the
//           stream never waits out a memory latency at a row boundary.
//           A token is kept only when its logit reaches the row's bound
//           L: a value that at least k logits of the row reach, so that
//           nothing below it can be in the top-k.  The eight warps raise L
//           together.  Every kept logit is counted in a histogram of the
//           row that the CTA shares (2048 bins: sign, exponent and the top
//           two mantissa bits of the logit), and L is the lower edge of
//           the highest bin at and above which k logits have been counted.
//           After the first few thousand tokens L sits just below the
//           row's k-th best logit and most steps of 512 tokens keep
//           nothing.  A buffer that fills (L held low by ties or by a
//           narrow spread of logits) is first cleared of entries below L,
//           then cut to its exact top-k; from then on the warp keeps only
//           logits above the k-th best it holds (later tokens have higher
//           ids, so an equal logit ranks below it).
//   merge   the ninth warp concatenates the eight segment lists (segment
//           order = token order), cuts them to the row's exact top-k and
//           writes the list and (m, Z), while the streaming warps go on to
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
// narrowing histograms, keeps the keys above K*, and the first (lowest-id)
// entries equal to K* up to k in all.
#pragma once

#include "sv_rowpass.cuh"

namespace sv {

constexpr int kTkWarps = 8;                       // streaming warps, one segment of the row each
constexpr int kTkThreads = (kTkWarps + 1) * 32;   // and the merging warp
constexpr int kTkCtasPerSm = 2;                   // resident CTAs per SM (launch bounds)
constexpr int kTkEpl = 16;                        // logits per lane per step
constexpr int kTkStep = 32 * kTkEpl;              // tokens per warp step
constexpr int kTkCap = kTkStep + SV_MAX_TOPK;     // candidates a streaming warp holds: a
                                                  // whole step fits after an exact cut
constexpr int kTkStageBytes = 2048;               // one bulk copy
constexpr int kTkStages = 3;                      // bulk copies in flight per streaming warp
constexpr int kTkSegAlign = 64;                   // segment starts: multiples of 64 tokens
constexpr int kTkBins = 2048;                     // the row histogram
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
// histogram bin of a key: sign, exponent and two mantissa bits
__device__ __forceinline__ int tk_bin_shift(int es) { return es == 2 ? 5 : 21; }
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

// Cut keys/ids [0, cnt) (token order, cnt > k) to their exact top-k, in
// place and in token order; returns (entries kept, K*).  K*, the k-th
// largest key, by narrowing a window of keys that holds it: starting from
// [min key, max key], a 256-bin histogram of the keys in the window (bins
// 2^shift wide, so the window fills the bins), walked down from the top bin
// until the running count reaches the rank still wanted, fixes the bin that
// holds K*; the next window is that bin.  The window adapts to how the
// held keys crowd together rather than following fixed digits; lanes that
// hit the same bin add once (warp-aggregated), so a crowded bin costs no
// serialised atomics.
__device__ __noinline__ uint2 tk_cut(unsigned* key, int* id, unsigned* hist, int cnt, int k,
                                     int lane) {
  __syncwarp();
  unsigned mn = 0xffffffffu, mx = 0u;
  for (int i = lane; i < cnt; i += 32) {
    mn = min(mn, key[i]);
    mx = max(mx, key[i]);
  }
  unsigned base = __reduce_min_sync(0xffffffffu, mn);
  unsigned span = __reduce_max_sync(0xffffffffu, mx) - base;  // the window: [base, base + span]
  unsigned need = static_cast<unsigned>(k);  // rank of K* within the window, from the top
  for (;;) {
    const int shift = span < 256u ? 0 : 24 - __clz(span);  // (span >> shift) < 256
#pragma unroll
    for (int q = 0; q < 8; ++q) hist[lane * 8 + q] = 0u;
    __syncwarp();
    for (int i0 = 0; i0 < cnt; i0 += 32) {
      const int i = i0 + lane;
      const unsigned kk = i < cnt ? key[i] : 0u;
      const bool in = i < cnt && kk >= base && kk - base <= span;
      const unsigned bin = in ? (kk - base) >> shift : 0u;
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
    __syncwarp();
    const unsigned lo_key = base + (static_cast<unsigned>(bin) << shift);
    if (shift == 0) {
      base = lo_key;
      break;
    }
    span = min((1u << shift) - 1u, span - (static_cast<unsigned>(bin) << shift));
    base = lo_key;
  }
  const unsigned kstar = base;  // need = how many entries equal to K* to keep
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned written = 0, ties = 0;
  for (int b0 = 0; b0 < cnt; b0 += 32) {
    const int i = b0 + lane;
    const bool in = i < cnt;
    const unsigned kk = in ? key[i] : 0u;
    const int ii = in ? id[i] : 0;
    const bool tie = in && kk == kstar;
    const unsigned tmask = __ballot_sync(0xffffffffu, tie);
    const bool keep = in && (kk > kstar || (tie && ties + __popc(tmask & lt_mask) < need));
    const unsigned kmask = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // every lane has read its entry of this tile
    if (keep) {
      const unsigned p = written + __popc(kmask & lt_mask);  // <= i: never ahead of a read
      key[p] = kk;
      id[p] = ii;
    }
    written += __popc(kmask);
    ties += __popc(tmask);
    __syncwarp();
  }
  __syncwarp();
  return make_uint2(written, kstar);
}

// Drop the entries of keys/ids [0, cnt) below key lk, in place and in token
// order; returns the entries kept.
__device__ __forceinline__ int tk_compact(unsigned* key, int* id, int cnt, unsigned lk, int lane) {
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned written = 0;
  for (int b0 = 0; b0 < cnt; b0 += 32) {
    const int i = b0 + lane;
    const bool in = i < cnt;
    const unsigned kk = in ? key[i] : 0u;
    const int ii = in ? id[i] : 0;
    const bool keep = in && kk >= lk;
    const unsigned kmask = __ballot_sync(0xffffffffu, keep);
    __syncwarp();
    if (keep) {
      const unsigned p = written + __popc(kmask & lt_mask);
      key[p] = kk;
      id[p] = ii;
    }
    written += __popc(kmask);
    __syncwarp();
  }
  __syncwarp();
  return static_cast<int>(written);
}

// A streaming warp's state for the row (the same in every lane).
struct TkWarp {
  unsigned* key;  // buffer, token order
  int* id;
  unsigned* hist;  // scratch of the exact cut
  int cnt;
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

// Raise L from the row histogram: the lower edge of the highest bin b with
// at least k logits counted at or above it.  Counts only grow and every
// counted logit is in the row, so the edge is a valid bound whenever it is
// read.  Other warps move the count and the top bin at any time: lane 0
// reads them once for the warp, so that every lane takes the same path.
__device__ __forceinline__ void tk_refresh(TkWarp& w, const volatile unsigned* hist,
                                           const volatile unsigned* top,
                                           const volatile unsigned* count, int k, int es,
                                           int lane) {
  unsigned n_seen = 0u, top_b = 0u;
  if (lane == 0) {
    n_seen = *count;
    top_b = *top;
  }
  n_seen = __shfl_sync(0xffffffffu, n_seen, 0);
  top_b = __shfl_sync(0xffffffffu, top_b, 0);
  if (n_seen < static_cast<unsigned>(k)) return;
  const int shift = tk_bin_shift(es);
  const int floor_b = static_cast<int>(w.lk >> shift);  // no gain at or below the bound's bin
  int hi = static_cast<int>(top_b);
  unsigned carry = 0;
  while (hi > floor_b) {
    const int b = hi - lane;
    const unsigned c = b > floor_b ? hist[b] : 0u;
    const unsigned incl = warp_incl_scan_u(c, lane) + carry;
    const unsigned hit = __ballot_sync(0xffffffffu, b > floor_b && incl >= static_cast<unsigned>(k));
    if (hit) {
      w.lk = static_cast<unsigned>(hi - (__ffs(hit) - 1)) << shift;
      tk_filter(w, es);
      return;
    }
    carry = __shfl_sync(0xffffffffu, incl, 31);
    hi -= 32;
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
  static constexpr int kFw = 32 / kG;       // bits per group in a packed count
};

// the j-th logit of group g (j warp-divergent; g a constant once the loop
// over groups is unrolled): selects, no local memory
template <int ES>
__device__ __forceinline__ float tk_pick(const float (&x)[kTkEpl], int g, int j) {
  const int o = g * TkStep<ES>::kEpg;
  if constexpr (TkStep<ES>::kEpg == 8) {
    const bool b0 = j & 1;
    const float a = b0 ? x[o + 1] : x[o], b = b0 ? x[o + 3] : x[o + 2];
    const float c = b0 ? x[o + 5] : x[o + 4], d = b0 ? x[o + 7] : x[o + 6];
    const float e = (j & 2) ? b : a, f = (j & 2) ? d : c;
    return (j & 4) ? f : e;
  } else {
    const bool b0 = j & 1;
    const float a = b0 ? x[o + 1] : x[o], b = b0 ? x[o + 3] : x[o + 2];
    return (j & 2) ? b : a;
  }
}

// the pass mask of a step: bit g EPG + j for logit (g, j)
template <int ES>
__device__ __forceinline__ unsigned tk_pass(const TkWarp& w, const float (&x)[kTkEpl]) {
  unsigned pass = 0;
#pragma unroll
  for (int i = 0; i < kTkEpl; ++i) pass |= (x[i] > w.fv || x[i] == w.eqv) ? (1u << i) : 0u;
  return pass;
}
// per-group pass counts of a lane, packed kFw bits per group
template <int ES>
__device__ __forceinline__ unsigned tk_pack_counts(unsigned pass) {
  using S = TkStep<ES>;
  unsigned c = 0;
#pragma unroll
  for (int g = 0; g < S::kG; ++g)
    c |= static_cast<unsigned>(__popc((pass >> (g * S::kEpg)) & ((1u << S::kEpg) - 1u))) << (g * S::kFw);
  return c;
}
template <int ES>
__device__ __forceinline__ unsigned tk_sum_fields(unsigned c) {
  using S = TkStep<ES>;
  unsigned t = 0;
#pragma unroll
  for (int g = 0; g < S::kG; ++g) t += (c >> (g * S::kFw)) & ((1u << S::kFw) - 1u);
  return t;
}

// Keep the logits of one step (x[i] for the bits of `valid`; the step
// starts at token id0) that pass the filter, appending them in token order
// (group by group, lanes in order within a group) and counting them in the
// row histogram; then raise L.  A full buffer is cleared of entries below L
// first, and cut to its exact top-k if that is not enough.
template <int ES>
__device__ __forceinline__ void tk_take(TkWarp& w, const float (&x)[kTkEpl], unsigned valid,
                                        int id0, int k, unsigned* rhist, unsigned* rtop,
                                        unsigned* rcount, int lane) {
  using S = TkStep<ES>;
  unsigned pass = tk_pass<ES>(w, x) & valid;
  unsigned cpk = tk_pack_counts<ES>(pass);
  unsigned incl = warp_incl_scan_u(cpk, lane);
  unsigned tot = __shfl_sync(0xffffffffu, incl, 31);
  unsigned total = tk_sum_fields<ES>(tot);
  if (total == 0u) return;
  if (w.cnt + static_cast<int>(total) > kTkCap) {
    w.cnt = tk_compact(w.key, w.id, w.cnt, w.lk, lane);
    if (w.cnt + static_cast<int>(total) > kTkCap) {
      const uint2 r = tk_cut(w.key, w.id, w.hist, w.cnt, k, lane);  // cnt > kTkStep > k
      w.cnt = static_cast<int>(r.x);
      w.thr = r.y;
      tk_filter(w, ES);
      pass = tk_pass<ES>(w, x) & valid;
      cpk = tk_pack_counts<ES>(pass);
      incl = warp_incl_scan_u(cpk, lane);
      tot = __shfl_sync(0xffffffffu, incl, 31);
      total = tk_sum_fields<ES>(tot);
      if (total == 0u) return;
    }
  }
  constexpr int shift = ES == 2 ? 5 : 21;
  const unsigned excl = incl - cpk;
  unsigned base = static_cast<unsigned>(w.cnt);
  unsigned mb = 0u;
#pragma unroll
  for (int g = 0; g < S::kG; ++g) {
    constexpr unsigned fm = (1u << S::kFw) - 1u;
    unsigned slot = base + ((excl >> (g * S::kFw)) & fm);
    unsigned pg = (pass >> (g * S::kEpg)) & ((1u << S::kEpg) - 1u);
    const int gid = id0 + g * S::kSpan + lane * S::kEpg;
    while (pg) {
      const int j = __ffs(pg) - 1;
      pg &= pg - 1u;
      const unsigned kk = tk_key_of(tk_pick<ES>(x, g, j), ES);
      w.key[slot] = kk;
      w.id[slot] = gid + j;
      ++slot;
      const unsigned b = kk >> shift;
      atomicAdd(rhist + b, 1u);
      mb = max(mb, b);
    }
    base += (tot >> (g * S::kFw)) & fm;
  }
  w.cnt += static_cast<int>(total);
  mb = __reduce_max_sync(0xffffffffu, mb);
  if (lane == 0) {
    atomicMax(rtop, mb);
    atomicAdd(rcount, total);
  }
  __syncwarp();
  tk_refresh(w, rhist, rtop, rcount, k, ES, lane);
}

// One step from its raw words (group g in raw[g]; logits beyond the segment
// are -inf and left out of `valid`).  The NaN-propagating maximum tells
// whether any logit can pass and, accumulated in mx, whether the row holds
// NaN or +inf.
template <int ES>
__device__ __forceinline__ void tk_step(TkWarp& w, const uint4 (&raw)[ES], unsigned valid,
                                        int id0, int k, unsigned* rhist, unsigned* rtop,
                                        unsigned* rcount, float& mx, int lane) {
  float m;
  if constexpr (ES == 2) {
    const unsigned m2 = bf16x2_max_nan(
        bf16x2_max_nan(bf16x2_max_nan(raw[0].x, raw[0].y), bf16x2_max_nan(raw[0].z, raw[0].w)),
        bf16x2_max_nan(bf16x2_max_nan(raw[1].x, raw[1].y), bf16x2_max_nan(raw[1].z, raw[1].w)));
    m = fmax_nan(bf16lo(m2), bf16hi(m2));
  } else {
    float q[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
      q[g] = fmax_nan(fmax_nan(__uint_as_float(raw[g].x), __uint_as_float(raw[g].y)),
                      fmax_nan(__uint_as_float(raw[g].z), __uint_as_float(raw[g].w)));
    m = fmax_nan(fmax_nan(q[0], q[1]), fmax_nan(q[2], q[3]));
  }
  mx = fmax_nan(mx, m);
  const bool hit = !(m <= w.fv) || m == w.eqv;
  if (!__any_sync(0xffffffffu, hit)) return;
  float x[kTkEpl];
#pragma unroll
  for (int g = 0; g < ES; ++g) {
    const unsigned v[4] = {raw[g].x, raw[g].y, raw[g].z, raw[g].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if constexpr (ES == 2) {
        x[g * 8 + 2 * h] = bf16lo(v[h]);
        x[g * 8 + 2 * h + 1] = bf16hi(v[h]);
      } else {
        x[g * 4 + h] = __uint_as_float(v[h]);
      }
    }
  }
  tk_take<ES>(w, x, valid, id0, k, rhist, rtop, rcount, lane);
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
  int n_stages;       // stages per row (the segment, 2 KB at a time)
  int seg_bytes;      // bytes of the segment
  int64_t seg_off;    // byte offset of the segment within a row
  unsigned issued, consumed;
};

__device__ __forceinline__ void tk_feed_issue(TkFeed& f, const TopkPass& a, int G, int n_rows) {
  if (f.row >= n_rows || f.n_stages == 0) return;
  const int slot = static_cast<int>(f.issued % kTkStages);
  const int off = f.stage * kTkStageBytes;
  const uint32_t bytes = static_cast<uint32_t>(min(kTkStageBytes, f.seg_bytes - off));
  fence_proxy_async_shared();  // the slot's earlier reads before the copy's writes
  mbar_arrive_expect_tx(&f.bar[slot], bytes);
  bulk_copy_g2s_hint(f.ring + slot * kTkStageBytes, tk_row_ptr(a, f.row) + f.seg_off + off, bytes,
                     &f.bar[slot], f.pol);
  ++f.issued;
  if (++f.stage == f.n_stages) {
    f.stage = 0;
    f.row = tk_next_row(a, f.row + G, G, n_rows);
  }
}

// The merging warp: the row's exact top-k from the eight segment lists of
// set p, the list and (m, Z) written out.  The lists are first packed
// together in place (segment order = token order).
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
  if (cnt > k) cnt = static_cast<int>(tk_cut(key, id, sh.cut_hist[kTkWarps], cnt, k, lane).x);
  __syncwarp();
  const bool bad = __shfl_sync(0xffffffffu, lane == 0 ? sh.bad[p] : 0u, 0) != 0u;
  float2* out = a.lists + static_cast<size_t>(r) * a.max_topk;
  float m = kNegInf;
  for (int i = lane; i < k; i += 32) {
    const bool in = i < cnt;
    const float v = in ? tk_value(key[i], a.es) : kNegInf;
    out[i] = make_float2(v, __int_as_float(in ? id[i] : -1));
    m = fmaxf(m, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const Scale2 c = scale_for(a.temperature[b]);
  float z = 0.f;
  if (m != kNegInf)
    for (int i = lane; i < cnt; i += 32) z += fast_exp2(scaled_arg(tk_value(key[i], a.es), m, c));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) {
    a.mz[r] = bad ? make_float2(__int_as_float(0x7fc00000), 0.f) : make_float2(m, z);
    sh.bad[p] = 0u;
  }
  __syncwarp();
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
  unsigned* rhist = sh.row_hist;
  // the histogram starts clear: each warp clears its eighth
  for (int i = warp * (kTkBins / kTkWarps) + lane; i < (warp + 1) * (kTkBins / kTkWarps); i += 32)
    rhist[i] = 0u;
  if (warp == 0 && lane == 0) {
    sh.top = 0u;
    sh.count = 0u;
  }
  TkFeed f;
  f.ring = &sh.ring[warp][0][0];
  f.bar = sh.ring_bar[warp];
  f.pol = policy_evict_first();
  f.seg_bytes = n * ES;
  f.seg_off = static_cast<int64_t>(s0) * ES;
  f.n_stages = a.bulk ? (f.seg_bytes + kTkStageBytes - 1) / kTkStageBytes : 0;
  f.row = tk_next_row(a, static_cast<int>(blockIdx.x), G, n_rows);
  f.stage = 0;
  f.issued = 0u;
  f.consumed = 0u;
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
    w.cnt = 0;
    w.lk = 0u;
    w.thr = 0u;
    tk_filter(w, ES);
    float mx = kNegInf;
    if (a.bulk) {
      for (int st = 0; st < f.n_stages; ++st) {
        const int slot = static_cast<int>(f.consumed % kTkStages);
        const uint32_t parity = (f.consumed / kTkStages) & 1u;
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
            tk_step<ES>(w, raw, valid, s0 + eb, k, rhist, &sh.top, &sh.count, mx, lane);
          }
        }
        __syncwarp();  // every lane is done with the slot
        ++f.consumed;
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
        tk_step<ES>(w, raw, valid, s0 + eb, k, rhist, &sh.top, &sh.count, mx, lane);
      }
    }
    const bool bad = mx != mx || mx == kPosInf;
    tk_refresh(w, rhist, &sh.top, &sh.count, k, ES, lane);
    w.cnt = tk_compact(w.key, w.id, w.cnt, w.lk, lane);
    if (w.cnt > k) w.cnt = static_cast<int>(tk_cut(w.key, w.id, w.hist, w.cnt, k, lane).x);
    // hand the segment's list over (set p is free once the row two back is merged)
    __syncwarp();
    named_sync(kTkBarFree + p, kTkThreads);
    for (int i = lane; i < w.cnt; i += 32) {
      sh.list_key[p][warp * SV_MAX_TOPK + i] = w.key[i];
      sh.list_id[p][warp * SV_MAX_TOPK + i] = w.id[i];
    }
    if (lane == 0) {
      sh.list_cnt[p][warp] = w.cnt;
      if (bad) sh.bad[p] = 1u;
    }
    named_arrive(kTkBarFull + p, kTkThreads);
    // every streaming warp is done with the row's histogram: clear it
    named_sync(kTkBarStream, kTkWarps * 32);
    for (int i = warp * (kTkBins / kTkWarps) + lane; i < (warp + 1) * (kTkBins / kTkWarps); i += 32)
      rhist[i] = 0u;
    if (warp == 0 && lane == 0) {
      sh.top = 0u;
      sh.count = 0u;
    }
    __syncwarp();
    named_sync(kTkBarStream, kTkWarps * 32);
    r = tk_next_row(a, r + G, G, n_rows);
  }
  // after a timeout, copies may still be in flight into the ring: wait for
  // them (briefly) before the CTA's shared memory is released
  if (lane == 0)
    for (; f.consumed < f.issued; ++f.consumed)
      mbar_wait_bounded(&f.bar[f.consumed % kTkStages], (f.consumed / kTkStages) & 1u,
                        kWaitLimitAfterTimeoutNs);
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
