// sv_rowpass.cuh -- definitions shared by the verification kernels: the
// CTA layout, shared-memory state, workspace view, chunk reductions and the
// inverse-CDF draw.
//
// Work is a flat list of "items"; an item is one 32 KB chunk of one logit
// row that the step must read (target rows 0..nd and, for sampled requests,
// draft rows 0..nd-1).  A producer warp claims items and moves each into a
// 4-stage shared-memory ring with a 1-D bulk copy (the TMA engine);
// consumer warps reduce the chunk -- (max, sum of exp) for sampled rows,
// (max, lowest argmax) for greedy rows -- and hand per-warp partials to a
// bookkeeper warp through a result ring; the bookkeeper combines them,
// stores one partial per chunk and counts per-request tickets; a finalizer
// group runs the finalize of each request whose last chunk is in (accept
// scan, emitted token) while the consumers keep streaming.  Every hand-off
// inside a CTA is an mbarrier; no CTA ever waits for another.
#pragma once

#include <stddef.h>

#include "sv_device.cuh"

namespace sv {

constexpr int kStages = 4;
constexpr int kChunkBytes = 32768;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kGroups = 2;                    // consumer groups, taking alternate chunks
constexpr int kGroupWarps = kConsumerWarps / kGroups;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kVecPerThread = kChunkBytes / 16 / kGroupThreads;  // 16-byte vectors per chunk
constexpr int kResSlots = 16;                 // result ring (consumers -> bookkeeper)
constexpr int kFinWarps = 4;                  // finalizer group
constexpr int kFinThreads = kFinWarps * 32;
// Warp roles.  The control warps come first: the warp schedulers favour
// lower warp ids among ready warps, and the consumers are ready almost
// always, so control work placed after them would wait for gaps.
constexpr int kProducerBase = 0;              // the producer warp
constexpr int kBkBase = 32;                   // bookkeeper warp
constexpr int kTkBase = 64;                   // ticket warp
constexpr int kFinBase = 96;                  // finalizer group (problems with draws: the
                                              // last of its warps is the draw scout)
constexpr int kScBase = kFinBase + 3 * 32;    // draw scout warp (problems with draws)
constexpr int kConsBase = kFinBase + kFinThreads;  // consumer warps
constexpr int kThreads = kConsBase + kConsumers;
constexpr int kRSeg = 256;                   // draw pass: tokens per segment (8 per lane)
constexpr int kPageSeg = 512;                // draw finalize: segments per page (16 per lane)
constexpr int kMaxPages = 8;                 // => at most 4096 segments (V <= 2^20)
constexpr int kFinCap = 128;                  // requests awaiting their finalize
constexpr int kBqCap = 256;                   // booked chunks awaiting their ticket
constexpr int kMbCap = 4;                     // planned draw chunks awaiting the producer
constexpr int kSegEl = 1024;        // inverse-CDF segment: 32 lanes x 32 elements
constexpr int kMaxSeg = 1024;       // => V <= 2^20
constexpr int kMaxRowsPerReq = 128;  // chain: 2K+1 <= 65; tree: N + M <= 128
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr uint64_t kWaitLimitAfterTimeoutNs = 1000000ull;  // 1 ms

static_assert(kVecPerThread * 16 * kGroupThreads == kChunkBytes, "chunk split");
static_assert(kStages % kGroups == 0, "each group owns whole stages");
static_assert(kVecPerThread == 4 || kVecPerThread == 8, "the bf16 reduction's sum tree");
// draw pass: 256-token segments per consumer warp and chunk
constexpr int kSpwBf16 = kChunkBytes / 2 / 2 / kRSeg / kGroupWarps;
constexpr int kSpwF32 = kChunkBytes / 2 / 4 / kRSeg / kGroupWarps;
static_assert(kSpwF32 >= 1 && kSpwBf16 <= 4, "draw-pass segments per warp");

enum RowKind : int { KIND_ARGMAX = 0, KIND_SOFTMAX = 1, KIND_TOPK = 2, KIND_RESID_PASS = 3 };

constexpr int kFinResid = 0x40000000;  // finalize-list flag: a residual draw (request id below)
constexpr int kDrawTicketBase = 1024;  // draw tickets follow the request tickets (SV_MAX_B)

struct WsHeader {
  unsigned int pad0[2];
  int error;
  unsigned int pad[5];
};

// Device view of the caller's workspace.
struct Ws {
  WsHeader* hdr;
  unsigned int* tickets;  // [2 SV_MAX_B] chunk counters: requests, then their draws
  float2* partials;       // [rows_max * ipr] one (max, sum) / (max, argmax) per chunk
  float* segsums;         // [B * ipr2 * segments per chunk] residual segment sums
  float* scratch;         // per-request residual rows (tree walk) [B][2][V]
  void* jobs;             // residual draws [SV_MAX_B][kJobWords]
};

// A residual / bonus draw (CMU 15-779 Lecture 17, sec. 2.3-2.4): request b,
// position n, mode 0: w = max(0, p_n - q_n), mode 1: w = p_n; the row
// statistics of p_n and q_n, and the temperature scale.
struct P2Job {
  int b, n, mode;
  int pos;  // the request's position in the processing order
  float mp, izp, mq, izq;
  float c_hi, c_lo;
};

// A published draw as the workspace holds it: kJobWords 64-bit words per
// request, each never zero once written, so the draw-pass scouts poll the
// words themselves -- no flag, no fence.
//   w0 = bits(1/Z_p) | bits(m_p) << 32      1/Z_p in (0, 1]: low word nonzero
//   w1 = bits(1/Z_q) | bits(m_q) << 32      low word 0x80000000 when unused
//   w2 = (1 + n + (mode << 8)) | failed << 32
// The temperature scale is not stored: every CTA holds it per position.
constexpr int kJobWords = 4;  // three used, one spare (32 bytes per request)

// Draw-pass segment sums are kept sign-flipped in the workspace: a sum is
// >= 0 (negative zero is stored as +0), so a stored sum is never the zero
// word, and zero marks a sum not yet written this call.
__device__ __forceinline__ unsigned enc_seg(float s) {
  const unsigned u = __float_as_uint(s);
  return (u == 0x80000000u ? 0u : u) ^ 0x80000000u;
}
__device__ __forceinline__ float dec_seg(unsigned w) { return __uint_as_float(w ^ 0x80000000u); }

struct StageMeta {
  int item;      // -1: no more work
  int pos;       // request position in processing order (main pass)
  int kind;
  int n_el;      // elements in this chunk
  int el_base;   // first element's index within the row
  float c_hi, c_lo;
  const char* src;   // first element of the chunk
  const char* src2;  // second row's chunk (residual pass), or null
  float4 aux;        // residual pass: mp, 1/Zp, mq, 1/Zq
  int sub;           // residual pass: mode
  int slot;          // where the chunk's partial / segment sums go
};

// What the bookkeeper needs about a result slot.
struct __align__(16) ResMeta {
  int item;      // -1: no more work
  int kind;
  int slot;      // where the chunk's partial(s) go
  int tkt;       // ticket (request id)
  int need;      // ticket value that completes the request / draw
  int fin_code;  // finalize-list entry on completion
  float c_hi, c_lo;
};

// A planned chunk as the producer lane that planned it holds it: the stage
// and result metadata, stored into the ring with 16-byte stores.
union PlanRec {
  struct {
    StageMeta m;
    ResMeta r;
  } s;
  uint4 v[(sizeof(StageMeta) + sizeof(ResMeta)) / 16];
};
static_assert(sizeof(StageMeta) % 16 == 0 && sizeof(ResMeta) == 32, "metadata in 16-byte words");
constexpr int kStageWords = sizeof(StageMeta) / 16;
constexpr int kResWords16 = sizeof(ResMeta) / 16;

struct FinScratch {
  double dsum[kFinWarps];
  float seg[kMaxSeg];
  float rm[kMaxRowsPerReq];
  float rz[kMaxRowsPerReq];
  int ridx[kMaxRowsPerReq];
  double base;
  int seg_k;
  int seg_mode;  // 0 normal, 1 take the last positive weight, 2 no mass
  int n_acc;
  int err;
  int token;
  int misc[8];
};

// Row statistics of one request, private to one finalizer warp.
struct WarpFin {
  float rm[kMaxRowsPerReq];
  float rz[kMaxRowsPerReq];
  int ridx[kMaxRowsPerReq];
};

struct __align__(16) Shared {
  uint64_t full[kStages];      // producer -> consumers: chunk landed (tx bytes)
  uint64_t empty[kStages];     // consumers -> producer: chunk in registers
  uint64_t res_done[kResSlots];  // producer meta + consumer partials -> bookkeeper
  uint64_t res_free[kResSlots];  // bookkeeper -> producer: slot consumed
  StageMeta meta[kStages];
  ResMeta res_meta[kResSlots];
  float4 res_part[kResSlots][kGroupWarps];
  unsigned p_it;               // next ring position (producer lanes, in turn)
  int4 bq[kBqCap];             // booked chunks: ticket, count that completes it, finalize code
  unsigned bq_tail;            // entries published (bookkeeper only)
  unsigned bq_head;            // entries ticketed (ticket warp only)
  unsigned tk_done;            // the ticket warp has ticketed every chunk
  int fin_q[kFinCap];
  unsigned fin_claim;          // finalize-list entries taken (finalizer warps, CAS)
  unsigned fin_tail;           // entries published (ticket warp only)
  unsigned fin_busy;           // finalizer warps inside a finalize
  unsigned bk_done;            // the bookkeeper has booked every chunk
  int fin_cmd;                 // group finalize command: pos, -1 idle, -2 exit
  int n_pos;
  int n_draw_cap;   // at most this many draws can be published (sampled requests)
  int timed_out;  // a bounded wait of this CTA expired: later waits are short
  FinScratch fin;
  WarpFin wfin[kFinWarps];
  PlanRec mb[kMbCap];          // scout -> producer: planned draw chunks
  unsigned mb_tail;            // records published (scout only)
  unsigned mb_head;            // records taken (producer only)
  unsigned sc_done;            // the scout has no more claims
};

// Bytes of Shared that a problem uses: the draw mailbox, at the end, only
// for problems with draw passes.
template <class P>
__host__ __device__ constexpr size_t shared_bytes() {
  return P::kHasDraws ? sizeof(Shared) : offsetof(Shared, mb);
}

// Per-position tables that follow Shared in dynamic shared memory.
struct PosTables {
  int* info;      // request id | kind << 16 | extra << 20
  int* rstart;    // [n_pos + 1] first flat row of each position
  float2* scale;  // log2(e)/t pair per position
  float4* aux;    // problem-specific per-position data (P::kAuxBytes each)
};

__device__ __forceinline__ int info_req(int info) { return info & 0xffff; }
__device__ __forceinline__ int info_kind(int info) { return (info >> 16) & 3; }
__device__ __forceinline__ int info_extra(int info) { return (info >> 20) & 0x7ff; }
__device__ __forceinline__ int make_info(int b, int kind, int extra) {
  return b | (kind << 16) | (extra << 20);
}

// Kind of a chain request from its scalar arguments (nd drafts, temperature
// t, top-k tk): KIND_ARGMAX for t == 0, KIND_TOPK for a filter that keeps
// fewer than V tokens (0 < tk < V, within the call's bound max_topk),
// KIND_SOFTMAX otherwise; -1 for invalid arguments (nd outside [0, K], t
// negative or NaN, tk negative or above max_topk, no draft rows for a
// sampled request with drafts).
__device__ __forceinline__ int chain_kind(int nd, float t, int tk, int K, int V, int max_topk,
                                          bool has_draft) {
  if (nd < 0 || nd > K || !(t >= 0.f) || tk < 0) return -1;
  if (t == 0.f) return KIND_ARGMAX;
  if (!has_draft && nd > 0) return -1;
  if (tk > 0 && tk < V) return tk <= max_topk ? KIND_TOPK : -1;
  return KIND_SOFTMAX;
}

// log2(e)/t as a float pair computed with fp32 divisions only: hi is the
// quotient rounded down, lo the quotient of the exact (non-negative)
// remainder.  Both parts are positive, so a -inf logit scales to -inf in
// both products and never meets +inf.
__device__ __forceinline__ Scale2 scale_for(float t) {
  const float l_hi = 1.44269502162933349609375f;     // fl(log2 e)
  const float l_lo = 1.925963033500011079e-08f;      // log2 e - l_hi
  Scale2 c;
  if (!(t > 0.f)) {
    c.hi = 0.f;
    c.lo = 0.f;
    return c;
  }
  c.hi = __fdiv_rd(l_hi, t);
  const float rem = fmaf(-c.hi, t, l_hi);
  c.lo = fmaxf(__fdiv_rn(rem + l_lo, t), 1.0e-45f);
  return c;
}

// Block-wide (all kThreads) exclusive scan of int4 values.
__device__ __forceinline__ int4 block_excl_scan4(int4 v, int4* warp_tot, int4& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int4 y;
    y.x = __shfl_up_sync(0xffffffffu, inc.x, o);
    y.y = __shfl_up_sync(0xffffffffu, inc.y, o);
    y.z = __shfl_up_sync(0xffffffffu, inc.z, o);
    y.w = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) {
      inc.x += y.x;
      inc.y += y.y;
      inc.z += y.z;
      inc.w += y.w;
    }
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  int4 before = make_int4(0, 0, 0, 0);
  total = make_int4(0, 0, 0, 0);
  for (int w = 0; w < kThreads / 32; ++w) {
    const int4 t = warp_tot[w];
    if (w < warp) {
      before.x += t.x;
      before.y += t.y;
      before.z += t.z;
      before.w += t.w;
    }
    total.x += t.x;
    total.y += t.y;
    total.z += t.z;
    total.w += t.w;
  }
  __syncthreads();
  return make_int4(before.x + inc.x - v.x, before.y + inc.y - v.y, before.z + inc.z - v.z,
                   before.w + inc.w - v.w);
}

// ------------------------------------------------------------ chunk reduce

__device__ __forceinline__ float nan_f() { return __int_as_float(0x7fc00000); }

// Fast path: bf16 chunk staged in shared memory.  Each consumer thread
// takes kVecPerThread 16-byte vectors, releases the stage as soon as they
// are in registers, then reduces them with independent accumulators.
template <int KIND>
__device__ __forceinline__ void reduce_chunk_bf16(const StageMeta& mt, const uint4* stage,
                                                  uint64_t* empty_bar, int ctid, int lane,
                                                  MS& ms, VI& vi) {
  const int nvec = mt.n_el >> 3;
  uint4 r[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int v = ctid + k * kGroupThreads;
    r[k] = v < nvec ? stage[v] : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);

  uint32_t mk[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k)
    mk[k] = bf16x2_max_nan(bf16x2_max_nan(r[k].x, r[k].y), bf16x2_max_nan(r[k].z, r[k].w));
  uint32_t mx2 = mk[0];
#pragma unroll
  for (int k = 1; k < kVecPerThread; ++k) mx2 = bf16x2_max_nan(mx2, mk[k]);
  const float a = bf16lo(mx2), b = bf16hi(mx2);
  float m = (a != a || b != b) ? nan_f() : fmaxf(a, b);
  if (m == kPosInf) m = nan_f();

  if (KIND == KIND_SOFTMAX) {
    float s = 0.f;
    if (m == m && m != kNegInf) {
      const Scale2 c{mt.c_hi, mt.c_lo};
      float sk[kVecPerThread];
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const uint32_t w[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          acc += fast_exp2(scaled_arg(bf16lo(w[h]), m, c));
          acc += fast_exp2(scaled_arg(bf16hi(w[h]), m, c));
        }
        sk[k] = acc;
      }
      if constexpr (kVecPerThread == 8)
        s = ((sk[0] + sk[1]) + (sk[2] + sk[3])) + ((sk[4] + sk[5]) + (sk[6] + sk[7]));
      else
        s = (sk[0] + sk[1]) + (sk[2] + sk[3]);
    }
    ms = MS{m, s};
  } else {
    // lowest index of m: the first vector (ascending) whose maximum is m,
    // then the first of its eight elements equal to m
    int idx = 0x7fffffff;
    if (m == m) {
      int kk = -1;
#pragma unroll
      for (int k = kVecPerThread - 1; k >= 0; --k) {
        const int v = ctid + k * kGroupThreads;
        const float f = fmaxf(bf16lo(mk[k]), bf16hi(mk[k]));
        if (v < nvec && f == m) kk = k;
      }
      if (kk >= 0) {
        uint4 rv = r[0];
#pragma unroll
        for (int k = 1; k < kVecPerThread; ++k)
          if (kk == k) rv = r[k];
        const uint32_t w[4] = {rv.x, rv.y, rv.z, rv.w};
        int j = 7;
#pragma unroll
        for (int h = 3; h >= 0; --h) {  // descending, so the lowest match wins
          if (bf16hi(w[h]) == m) j = 2 * h + 1;
          if (bf16lo(w[h]) == m) j = 2 * h;
        }
        idx = mt.el_base + (ctid + kk * kGroupThreads) * 8 + j;
      }
    }
    vi = VI{m, idx};
  }
}

// Generic path: any dtype, chunk either staged (bulk) or read from global.
// Out of line, so the streaming loop's code stays compact.
template <int KIND>
__device__ __forceinline__ void reduce_chunk_generic(const StageMeta& mt, const char* stage,
                                                     bool staged, int es,
                                                     uint64_t* empty_bar, int ctid, int lane,
                                                     MS& ms, VI& vi) {
  const char* base = staged ? stage : mt.src;
  auto ld = [&](int e) -> float {
    if (es == 2) return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(base)[e]);
    return reinterpret_cast<const float*>(base)[e];
  };
  // ascending index within the thread: strict ">" keeps the lowest index
  float m = kNegInf;
  bool bad = false;
  int idx = 0x7fffffff;
  for (int e = ctid; e < mt.n_el; e += kGroupThreads) {
    const float x = ld(e);
    if (x != x || x == kPosInf) bad = true;
    if (idx == 0x7fffffff || x > m) {
      m = x;
      idx = mt.el_base + e;
    }
  }
  if (KIND == KIND_SOFTMAX) {
    float s = 0.f;
    if (!bad && m != kNegInf) {
      const Scale2 c{mt.c_hi, mt.c_lo};
      for (int e = ctid; e < mt.n_el; e += kGroupThreads) s += fast_exp2(scaled_arg(ld(e), m, c));
    }
    ms = bad ? MS{nan_f(), 0.f} : MS{m, s};
  } else {
    vi = bad ? VI{nan_f(), 0} : VI{m, idx};
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
}

// A logit-row chunk reduced by one consumer warp: (max, sum exp) for
// sampled rows, (max, lowest argmax) for greedy rows, warp-reduced.
__device__ __forceinline__ float2 reduce_row_chunk(const StageMeta& mt, const unsigned char* sp,
                                                   uint64_t* empty_bar, int ctid, int lane,
                                                   bool bulk, int es) {
  MS ms{kNegInf, 0.f};
  VI vi{kNegInf, 0x7fffffff};
  const bool fast = bulk && es == 2;
  if (mt.kind == KIND_ARGMAX) {
    if (fast)
      reduce_chunk_bf16<KIND_ARGMAX>(mt, reinterpret_cast<const uint4*>(sp), empty_bar, ctid,
                                     lane, ms, vi);
    else
      reduce_chunk_generic<KIND_ARGMAX>(mt, reinterpret_cast<const char*>(sp), bulk, es,
                                        empty_bar, ctid, lane, ms, vi);
    vi = warp_reduce_vi(vi);
    return make_float2(vi.v, __int_as_float(vi.i));
  }
  if (fast)
    reduce_chunk_bf16<KIND_SOFTMAX>(mt, reinterpret_cast<const uint4*>(sp), empty_bar, ctid,
                                    lane, ms, vi);
  else
    reduce_chunk_generic<KIND_SOFTMAX>(mt, reinterpret_cast<const char*>(sp), bulk, es,
                                       empty_bar, ctid, lane, ms, vi);
  ms = warp_reduce_ms(ms, Scale2{mt.c_hi, mt.c_lo});
  return make_float2(ms.m, ms.s);
}

// ------------------------------------------------------ residual weights

struct ResidParams {
  float mp, izp, mq, izq;
  Scale2 c;
  int mode;  // 0: max(0, p - q); 1: unnormalised p
};

// Residual weight of one token from its two logits.  Every operation is an
// explicitly rounded intrinsic, so the chunk pass and the final rescan
// produce the same bits.
__device__ __forceinline__ float resid_weight(float xp, float xq, const ResidParams& r) {
  // mp and mq are finite (a row whose maximum is not is an error and gets
  // no draw), so x = -inf gives d = -inf and a weight of 0
  const float dp = __fsub_rn(xp, r.mp);
  const float ep = fast_exp2(__fmaf_rn(dp, r.c.hi, __fmul_rn(dp, r.c.lo)));
  if (r.mode != 0) return ep;
  const float dq = __fsub_rn(xq, r.mq);
  const float eq = fast_exp2(__fmaf_rn(dq, r.c.hi, __fmul_rn(dq, r.c.lo)));
  return fmaxf(__fsub_rn(__fmul_rn(ep, r.izp), __fmul_rn(eq, r.izq)), 0.f);
}

__device__ __forceinline__ float warp_incl_scan_rn(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, y);
  }
  return x;
}

// ---------------------------------------------------------- inverse CDF

// Draw by inverse CDF from 32-element weight blocks produced by wf(i0, w)
// (w[j] = weight of token i0 + j, zero beyond V): the smallest t with
// u * S < C(t), C the running sum over ascending id, S the total; if
// rounding leaves none, the largest t with positive weight.  Sums: fp32
// within a lane (sequential) and across lanes (warp scan); fp64 across
// segments and for the final comparisons.  Called by all kConsumers
// threads; returns the token (-1 if S == 0) in every thread.
template <class WF>
__device__ int icdf_draw(int V, double u, const WF& wf, FinScratch& fs, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int nseg = (V + kSegEl - 1) / kSegEl;
  for (int s = warp; s < nseg; s += kFinWarps) {
    float w[32];
    wf(s * kSegEl + lane * 32, w);
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) ls += w[j];
    const float inc = warp_incl_scan(ls, lane);
    if (lane == 31) fs.seg[s] = inc;
  }
  named_sync(1, kFinThreads);
  if (warp == 0) {
    const int per = (nseg + 31) / 32;
    const int lo = min(lane * per, nseg), hi = min(lo + per, nseg);
    double lt = 0.0;
    for (int s = lo; s < hi; ++s) lt += static_cast<double>(fs.seg[s]);
    const double incl = warp_incl_scan_d(lt, lane);
    double excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0;
    const double S = __shfl_sync(0xffffffffu, incl, 31);
    const double target = u * S;
    int found = -1;
    double base = 0.0, run = excl;
    int last_pos = -1;
    for (int s = lo; s < hi; ++s) {
      const double nxt = run + static_cast<double>(fs.seg[s]);
      if (found < 0 && target < nxt) {
        found = s;
        base = run;
      }
      if (fs.seg[s] > 0.f) last_pos = s;
      run = nxt;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
    const unsigned pos = __ballot_sync(0xffffffffu, last_pos >= 0);
    if (lane == 0) {
      fs.seg_mode = 2;
      fs.seg_k = -1;
    }
    __syncwarp();
    if (!(S > 0.0)) {
      // no mass: mode 2
    } else if (hit) {
      const int src = __ffs(hit) - 1;
      if (lane == src) {
        fs.seg_k = found;
        fs.base = base;
        fs.seg_mode = 0;
      }
    } else if (pos) {
      const int src = 31 - __clz(pos);
      if (lane == src) {
        fs.seg_k = last_pos;
        fs.seg_mode = 1;
      }
    }
    __syncwarp();
    if (fs.seg_mode != 2) {
      const int k = fs.seg_k;
      float w[32];
      wf(k * kSegEl + lane * 32, w);
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) ls += w[j];
      const float inc = warp_incl_scan(ls, lane);
      float exl = __shfl_up_sync(0xffffffffu, inc, 1);
      if (lane == 0) exl = 0.f;
      int tok = -1;
      if (fs.seg_mode == 0) {
        const bool lane_hit = target < fs.base + static_cast<double>(inc);
        const unsigned lh = __ballot_sync(0xffffffffu, lane_hit);
        const int src = lh ? __ffs(lh) - 1 : 31;
        if (lane == src) {
          double c = fs.base + static_cast<double>(exl);
          int lastp = -1;
          for (int j = 0; j < 32; ++j) {
            c += static_cast<double>(w[j]);
            if (w[j] > 0.f) lastp = j;
            if (tok < 0 && target < c) tok = j;
          }
          if (tok < 0) tok = lastp;
          tok = tok < 0 ? -1 : k * kSegEl + lane * 32 + tok;
        }
        tok = __shfl_sync(0xffffffffu, tok, src);
      } else {
        int lastp = -1;
        for (int j = 0; j < 32; ++j)
          if (w[j] > 0.f) lastp = j;
        const unsigned lp = __ballot_sync(0xffffffffu, lastp >= 0);
        const int src = lp ? 31 - __clz(lp) : 0;
        tok = __shfl_sync(0xffffffffu, lastp < 0 ? -1 : k * kSegEl + lane * 32 + lastp, src);
      }
      if (lane == 0) fs.token = tok;
    } else if (lane == 0) {
      fs.token = -1;
    }
  }
  named_sync(1, kFinThreads);
  const int tok = fs.token;
  named_sync(1, kFinThreads);
  return tok;
}

// Load 32 consecutive logits [i0, i0+32) of a row as floats (0 beyond V is
// NOT applied here; `valid` counts the in-range ones).
__device__ __forceinline__ void load32(const char* row, int es, bool vec_ok, int i0, int V,
                                       float* x) {
  if (es == 2 && vec_ok && i0 + 32 <= V) {
    const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<size_t>(i0) * 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(p + q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[q * 8 + 2 * h] = bf16lo(w[h]);
        x[q * 8 + 2 * h + 1] = bf16hi(w[h]);
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int t = i0 + j;
    if (t < V) {
      x[j] = es == 2 ? bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(row) + t))
                     : __ldg(reinterpret_cast<const float*>(row) + t);
    } else {
      x[j] = kNegInf;
    }
  }
}

__device__ __forceinline__ float load_logit(const char* row, int es, int t) {
  return es == 2 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[t])
                 : reinterpret_cast<const float*>(row)[t];
}

// Eight consecutive logits [t0, t0 + 8) of a row piece holding n valid
// entries; entries at or beyond n read as -inf.  With vec the piece is
// 16-byte aligned and may be read in whole 16-byte vectors up to n rounded
// up to a vector (a staged chunk, or an aligned row of 16-byte multiple
// length); otherwise entries are read one by one.
__device__ __forceinline__ void load8(const char* base, int es, bool vec, int t0, int n,
                                      float* x) {
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = kNegInf;
  if (t0 >= n) return;
  if (vec && es == 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(t0) * 2);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      x[2 * h] = bf16lo(w[h]);
      x[2 * h + 1] = bf16hi(w[h]);
    }
  } else if (vec) {
    const float4 a = *reinterpret_cast<const float4*>(base + static_cast<size_t>(t0) * 4);
    x[0] = a.x;
    x[1] = a.y;
    x[2] = a.z;
    x[3] = a.w;
    if (t0 + 4 < n) {
      const float4 c = *reinterpret_cast<const float4*>(base + static_cast<size_t>(t0) * 4 + 16);
      x[4] = c.x;
      x[5] = c.y;
      x[6] = c.z;
      x[7] = c.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (t0 + j < n) x[j] = load_logit(base, es, t0 + j);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (t0 + j >= n) x[j] = kNegInf;
}

// Residual weights of eight tokens and their sequential fp32 sum; tokens at
// or beyond n weigh 0.  The draw pass and the final rescan both go through
// here, so they produce the same bits.
__device__ __forceinline__ float resid_weights8(const float* xp, const float* xq, int t0, int n,
                                                const ResidParams& r, float* w) {
  float ls = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    w[j] = t0 + j < n ? resid_weight(xp[j], xq[j], r) : 0.f;
    ls = __fadd_rn(ls, w[j]);
  }
  return ls;
}

}  // namespace sv
