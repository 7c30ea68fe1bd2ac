// Accept / reject / resample in one kernel on 4-CTA thread-block clusters.
//
// The method is the one of reject_sample.cu (page 1 §2.3, §4.1, §4.3; page 2
// §2.1-§2.2; page 3 formal definition and tree section): p = softmax(z/T),
// q = softmax(d/T); child x of node n is accepted iff u * Q(x) < P(x); a
// rejection turns the working target P into normalize(max(0, P - q)) and the
// next sibling is tried; a node whose children were all rejected, or a node
// without children, draws one token from its working P by inverse CDF in
// vocabulary order.  What differs is the schedule.
//
// Work item = one (request b, node n): the target row n, and the draft row n
// when n has children.  Every item is decided as if n were on the accepted
// path: its statistics, the tests of its children, and the draw at n when no
// child is accepted.  A request is finished when all its items are: the last
// one reads the items' records, walks the path from the root and writes the
// outputs.  Items whose parent is already known to be off the path skip
// their tests and draws (their rows are still read: every row of a request
// must hold a distribution).
//
// Each item is split over the four CTAs of a cluster, CTA r holding the
// r-th quarter of the row's 2048-logit chunks (1024 for fp32 logits).  The
// CTAs exchange per-quarter statistics through distributed shared memory, so
// each of them forms the same row normalisers, runs the same tests and makes
// the same choices.  Items are claimed in node-major order (all requests'
// roots, then all first children, ...), so an item's parent has usually been
// decided by the time the item is.
//
// Roles of the 16 warps of a CTA:
//   warp 0, lane 0  producer: 1-D bulk copies of chunks into a ring of 24
//                   8 KB slots (target chunk + draft chunk), in task order;
//                   statistics tasks of the claimed items, and the re-read
//                   tasks the control warp asks for (a residual pass over the
//                   quarter; one chunk for the in-chunk search);
//   warp 1          scheduler: rank 0 claims items (a global counter) and
//                   sends their indices to the four CTAs; each CTA loads the
//                   item's temperature, children and their tokens;
//   warp 2          control: exchanges, normalisers, tests, draw location,
//                   the item's record, the request's outputs;
//   warps 3..15     consumers: take the ring's tasks in order (task t on
//                   consumer t mod 13): chunk statistics, residual masses,
//                   in-chunk search.
// Every wait is bounded; a wait that gives up raises SPEC_ERR_TIMEOUT, tells
// the other CTAs of the cluster to stop, waits for the copies it issued and
// leaves with the cluster.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "philox.cuh"
#include "reject_sample.cuh"
#include "rs_device.cuh"
#include "tc_ptx.cuh"

namespace specv {
namespace rsf {

constexpr int kC = 4;              // CTAs per cluster: quarters of each row
constexpr int kThreads = 512;
constexpr int kSchedWarp = 1;
constexpr int kCtrlWarp = 2;       // first of the control warps
constexpr int kCtl = 6;            // control warps: items k, k + 6, ... go to control k mod 6
constexpr int kFirstConsumer = kCtrlWarp + kCtl;
constexpr int kConsumers = kThreads / kWarp - kFirstConsumer;  // 8
constexpr int kSlots = 20;         // ring slots
constexpr int kHalfSlot = 4096;    // one chunk of one row
constexpr int kSlotBytes = 2 * kHalfSlot;
constexpr int kNQ = 2 * kCtl;      // items in flight per CTA (two per control)
constexpr int kNE = 2;             // exchange buffers per control
constexpr int kMaxQuarter = 32;    // chunks per quarter
constexpr int kMaxKids = 63;
constexpr int kReqQ = 4;           // requests of one control to the producer

enum : int { kTaskStats = 0, kTaskRes = 1, kTaskSearch = 2, kTaskStop = 3 };
enum : int { kReqRes = 1, kReqSearch = 2 };
// record flags: the spec_status bits of a failed item (bits 0..7), the
// node's path state (bits 8..9: 0 off, 1 on, 2 unknown), bit 10: the node
// drew, bits 16..23: parent + 1
constexpr uint32_t kOnShift = 8, kDrewBit = 1u << 10, kParShift = 16;
constexpr uint32_t kPathOff = 0, kPathOn = 1, kPathUnknown = 2;

struct TaskDesc {
  int type, q, c, pad;
};

// The law a residual pass or an in-chunk search weighs elements by.
//   mode 0: w = 2^((z_t - mT) cs)                       (p, unnormalised)
//   mode 1: w = max(0, p - c q), p = 2^((z_t - mT) cs) / ST,
//                                q = 2^((z_d - mD) cs) / SD
struct Law {
  float mT, mD, invST, invSD, cs, c;
  int mode, pad;
};

struct ItemState {
  // filled by the scheduler
  int item;                 // -1: no more items
  int b, n, pair;           // request, node; pair: the node has children (its draft row is read)
  int nkids;
  uint32_t bad;             // spec_status bits found by the scheduler
  float cs;                 // log2(e) / T (1 for a greedy request)
  int greedy;               // temperature 0: every law is the point mass on the row's argmax
  int par;                  // parent node (-1 for the root)
  int kid[kMaxKids];        // children, ascending
  int ktok[kMaxKids];       // their drafted tokens
  // filled by the consumers
  RowStat st_t[kMaxQuarter], st_d[kMaxQuarter];
  float2 gz[kMaxKids];      // (target, draft) logit of each child's token, where this CTA has it
  unsigned long long have;  // bit j: gz[j] is set
  int s_done, r_done;
  double res[kMaxQuarter];  // residual masses of the quarter's chunks
  Law law;                  // set by the control before a residual pass or a search
  float trel_hi, trel_lo;   // search target inside the chunk (double-float)
  int s_tok;
  float s_w;
};

// One CTA's message of an exchange: the quarter's statistics (or, for a
// residual pass, its mass in s_t) and the children's logits it holds.
struct __align__(16) XMsg {
  float m_t, m_d;
  double s_t, s_d;
  unsigned long long have;
  uint32_t flags, path;
  int amax_t, amax_d;       // greedy: the quarter's first maximum (element index), -1 if none
  float2 gz[kMaxKids + 1];
};

// A drawn token, sent by the CTA that searched it to rank 0.
struct __align__(8) DrawMsg {
  int tok;
  float psamp;
};
__device__ __forceinline__ unsigned long long pack_draw(int tok, float psamp) {
  return ((unsigned long long)__float_as_uint(psamp) << 32) | (uint32_t)tok;
}

struct __align__(8) Bars {
  uint64_t full[kSlots], empty[kSlots];
  uint64_t meta[kNQ];     // local: the scheduler filled the item's state
  uint64_t bcast[kNQ];    // rank 0 sent the item index (1 arrival)
  uint64_t freed[kNQ];    // rank 0 only: the four controls are done with the slot
  uint64_t stats[kNQ], resd[kNQ], srch[kNQ];
  uint64_t drawn[kNQ];    // rank 0 only: the draw's result arrived
  uint64_t xbar[kCtl][kNE];
  int bcast_item[kNQ];
  DrawMsg draw[kNQ];
  TaskDesc task[kSlots];
  int req_type[kCtl][kReqQ], req_q[kCtl][kReqQ], req_c[kCtl][kReqQ];
  int req_tail[kCtl];
  int ctrl_done;          // controls that have finished
  int prod_items;         // items whose state the producer has taken (it may then be reused)
  int abort;
  uint32_t epoch_tag;
};

struct Rec {             // per (request, node) in the workspace, 32 bytes
  uint32_t done;         // the call's epoch tag once the item is finished
  uint32_t flags;
  int32_t acc_child;     // accepted child, -1 if none
  int32_t tok;           // the accepted child's token, else the drawn token
  float z, psamp;        // mass of the residual drawn from (1 for p), drawn token's probability
  float pc, qc;          // this node's own test, written by its parent's item (-1: not tested)
};
static_assert(sizeof(Rec) == 32, "record size");

constexpr size_t kRingOff = 0;
constexpr size_t kItemsOff = kRingOff + (size_t)kSlots * kSlotBytes;
constexpr size_t kXbufOff = kItemsOff + (((sizeof(ItemState) * kNQ) + 15) / 16) * 16;
constexpr size_t kBarsOff = kXbufOff + sizeof(XMsg) * kCtl * kNE * kC;
constexpr size_t kSmemBytes = kBarsOff + sizeof(Bars) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ void store4(float* p, float a, float b, float c, float e) {
  p[0] = a;
  p[1] = b;
  p[2] = c;
  p[3] = e;
}

__device__ __forceinline__ void store_rec_u32(Rec* r, int field, uint32_t v) {
  reinterpret_cast<volatile uint32_t*>(r)[field] = v;
}
__device__ __forceinline__ void store_rec_f32(Rec* r, int field, float v) {
  reinterpret_cast<volatile float*>(r)[field] = v;
}

// Element weights of 8 consecutive elements (one 16-byte vector per row),
// masked past `nvalid`.
template <typename T>
__device__ __forceinline__ float vec_law(const uint4& vt, const uint4& vd, int e, int nvalid,
                                         const Law& L, float (&w)[16 / sizeof(T)]) {
  constexpr int EPV = 16 / sizeof(T);
  float zt[EPV], zd[EPV];
  unpack16(vt, zt);
  unpack16(vd, zd);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPV; ++i) {
    float x;
    const float et = fast_exp2((zt[i] - L.mT) * L.cs);
    if (L.mode == 0) {
      x = et;
    } else {
      const float pv = et * L.invST;
      const float qv = fast_exp2((zd[i] - L.mD) * L.cs) * L.invSD;
      x = fmaxf(pv - L.c * qv, 0.f);
    }
    w[i] = (e + i < nvalid) ? x : 0.f;
    s += w[i];
  }
  return s;
}

__device__ __forceinline__ uint32_t word4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Inverse CDF inside one chunk held in shared memory, by one warp: lane l
// weighs its kStatVecs vectors, the lanes' sums are scanned as
// double-floats, the owning lane's words are spread over the warp and
// scanned again.  Returns the first element whose running weight exceeds
// trel, else the last of positive weight; *w_out = its weight.
template <typename T>
__device__ int smem_chunk_draw(const uint4* sv_t, const uint4* sv_d, int e0, int nvalid,
                               const Law& L, dfloat trel, float* w_out) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int E = kStatVecs * EPV;  // elements per lane
  constexpr int EW = 4 / sizeof(T);   // elements per 32-bit word
  const int lane = threadIdx.x % kWarp;
  uint4 rt[kStatVecs], rd[kStatVecs];
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v) {
    rt[v] = sv_t[lane * kStatVecs + v];
    rd[v] = L.mode == 1 ? sv_d[lane * kStatVecs + v] : make_uint4(0, 0, 0, 0);
  }
  float vs = 0.f;
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v) {
    float w[EPV];
    vs += vec_law<T>(rt[v], rd[v], lane * E + v * EPV, nvalid, L, w);
  }
  const dfloat incl = df_warp_scan(df_make(vs));
  const dfloat excl = df_sub(incl, df_make(vs));
  const unsigned hit =
      __ballot_sync(0xffffffffu, vs > 0.f && !df_gt(excl, trel) && df_gt(incl, trel));
  const unsigned pos = __ballot_sync(0xffffffffu, vs > 0.f);
  const int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
  const dfloat r = df_sub(trel, df_shfl(excl, owner));
  uint32_t wt = 0, wd = 0;  // lane l takes word l of the owner's elements
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t xt = __shfl_sync(0xffffffffu, word4(rt[v], i), owner);
      const uint32_t xd = __shfl_sync(0xffffffffu, word4(rd[v], i), owner);
      if (lane == v * 4 + i) {
        wt = xt;
        wd = xd;
      }
    }
  const int seg = owner * E;
  float w[EW];
  float ls = 0.f;
#pragma unroll
  for (int i = 0; i < EW; ++i) {
    float zt, zd;
    if (EW == 2) {
      zt = __uint_as_float(i == 0 ? wt << 16 : wt & 0xffff0000u);
      zd = __uint_as_float(i == 0 ? wd << 16 : wd & 0xffff0000u);
    } else {
      zt = __uint_as_float(wt);
      zd = __uint_as_float(wd);
    }
    const float et = fast_exp2((zt - L.mT) * L.cs);
    float x = et;
    if (L.mode == 1) x = fmaxf(et * L.invST - L.c * (fast_exp2((zd - L.mD) * L.cs) * L.invSD), 0.f);
    w[i] = (seg + lane * EW + i < nvalid) ? x : 0.f;
    ls += w[i];
  }
  const dfloat cum = df_warp_scan(df_make(ls));
  const dfloat before = df_sub(cum, df_make(ls));
  const unsigned h2 = __ballot_sync(0xffffffffu, ls > 0.f && df_gt(cum, r));
  const unsigned p2 = __ballot_sync(0xffffffffu, ls > 0.f);
  int k = 0;
  if (EW == 2) {
    if (h2) {
      k = (w[0] > 0.f && df_gt(df_add(before, df_make(w[0])), r)) ? 0 : 1;
      if (w[k] <= 0.f) k = 1 - k;
    } else {
      k = w[1] > 0.f ? 1 : 0;
    }
  }
  const int l2 = h2 ? __ffs(h2) - 1 : (p2 ? 31 - __clz(p2) : 0);
  const int tok = e0 + seg + lane * EW + k;
  const float wk = w[EW == 2 ? (k & 1) : 0];
  *w_out = __shfl_sync(0xffffffffu, wk, l2);
  return __shfl_sync(0xffffffffu, tok, l2);
}

// The quarter's statistics combined in fp64 (same order on every CTA).
__device__ __forceinline__ void quarter_stats(const RowStat* st, int nq, float cs, float* m_out,
                                              double* s_out) {
  float m = -INFINITY;
  for (int j = 0; j < nq; ++j) m = fmaxf(m, st[j].m);
  double s = 0.0;
  for (int j = 0; j < nq; ++j)
    if (st[j].m != -INFINITY || st[j].s != st[j].s) s += st[j].s * (double)fast_exp2((st[j].m - m) * cs);
  *m_out = m;
  *s_out = s;
}

// Row normaliser from the four quarters (rank order).
__device__ __forceinline__ void row_norm(const XMsg* x, bool draft, float cs, float* m_out,
                                         double* s_out) {
  float m = -INFINITY;
  for (int r = 0; r < kC; ++r) m = fmaxf(m, draft ? x[r].m_d : x[r].m_t);
  double s = 0.0;
  for (int r = 0; r < kC; ++r) {
    const float mr = draft ? x[r].m_d : x[r].m_t;
    const double sr = draft ? x[r].s_d : x[r].s_t;
    if (mr != -INFINITY || sr != sr) s += sr * (double)fast_exp2((mr - m) * cs);
  }
  *m_out = m;
  *s_out = s;
}

__device__ __forceinline__ bool norm_ok(float m, double s) {
  return m > -INFINITY && m < INFINITY && s > 0.0 && s < INFINITY;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) rs_fused_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parent, const float* __restrict__ temperature, uint64_t seed,
    uint64_t offset, uint64_t b_base, int32_t* __restrict__ out_tokens,
    int32_t* __restrict__ path, int32_t* __restrict__ accepted_len, float* __restrict__ probe,
    spec_dims d, int n_chunks, Rec* recs, uint32_t* req_done, uint32_t* ctl,
    uint32_t* status) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int CH = kWarp * kStatVecs * EPV;  // logits per chunk (4 KB of one row)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem + kRingOff;
  ItemState* items = reinterpret_cast<ItemState*>(smem + kItemsOff);
  XMsg* xbuf = reinterpret_cast<XMsg*>(smem + kXbufOff);  // [kCtl][kNE][kC]
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarsOff);

  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const uint32_t rank = ptx::cluster_rank();
  const int B = d.B, M = d.M, V = d.V;
  const int I = B * M;  // items
  const int cpq = (n_chunks + kC - 1) / kC;  // chunks per quarter
  const int q0 = min(n_chunks, (int)rank * cpq), q1 = min(n_chunks, q0 + cpq);
  const int nq = q1 - q0;  // this CTA's chunks of every row
  const uint64_t wait = wait_limit_cycles(d);
  uint32_t* item_counter = ctl;      // next item to claim
  uint32_t* ctas_done = ctl + 1;     // CTAs finished (the last resets the counters)
  uint32_t* epoch = ctl + 2;         // tag of the last finished call

  pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < kNQ; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->meta[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->bcast[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->freed[i]), kC);
      ptx::mbar_init(ptx::smem_u32(&bars->stats[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->resd[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->srch[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->drawn[i]), 1);
    }
    for (int j = 0; j < kCtl; ++j) {
      for (int i = 0; i < kNE; ++i) ptx::mbar_init(ptx::smem_u32(&bars->xbar[j][i]), kC);
      bars->req_tail[j] = 0;
    }
    bars->ctrl_done = 0;
    bars->prod_items = 0;
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::cluster_sync_all();  // every CTA's barriers exist before any remote arrival
  pdl_wait();               // inputs and the workspace counters come from earlier work
  if (tid == 0) {
    uint32_t tag = ld_volatile_u32(epoch) + 1u;
    bars->epoch_tag = tag == 0 ? 1u : tag;
  }
  __syncthreads();
  const uint32_t tag = bars->epoch_tag;
  volatile int* abort = &bars->abort;

  // tell the other CTAs of the cluster to stop too (their waits would give
  // up after their own limits anyway; this only makes it prompt)
  auto spread_abort = [&]() {
    for (uint32_t r = 0; r < kC; ++r)
      if (r != rank) ptx::st_cluster_u32(ptx::map_rank(ptx::smem_u32(&bars->abort), r), 1u);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int64_t task = 0;
      int k_item = 0;             // next local item to start
      bool items_done = false;
      int cur_q = -1, s_next = 0; // statistics tasks of the current item: chunks s_next..q1
      bool cur_pair = false;
      const T* cur_t = nullptr;
      const T* cur_d = nullptr;
      int head[kCtl];             // next request of each control warp
      for (int j = 0; j < kCtl; ++j) head[j] = 0;
      int rr = 0;                 // control whose queue is looked at first
      int rq_type = 0, rq_q = 0, rq_c = 0, rq_end = 0;
      bool ok = true;
      long long t_idle = 0;
      auto issue = [&](int type, int q, int c, const T* trow, const T* drow, bool need_d) -> bool {
        const int slot = (int)(task % kSlots);
        if (task >= kSlots &&
            !ptx::mbar_wait(ptx::smem_u32(&bars->empty[slot]), (uint32_t)(((task / kSlots) & 1) ^ 1),
                            abort, wait))
          return false;
        bars->task[slot] = TaskDesc{type, q, c, 0};
        const uint32_t fb = ptx::smem_u32(&bars->full[slot]);
        if (type == kTaskStop) {
          ptx::mbar_arrive(fb);
        } else {
          const int e0 = c * CH;
          const uint32_t bytes = (uint32_t)(min(CH, V - e0) * (int)sizeof(T));
          ptx::mbar_arrive_expect_tx(fb, need_d ? 2 * bytes : bytes);
          uint8_t* sp = ring + (size_t)slot * kSlotBytes;
          ptx::bulk_g2s(ptx::smem_u32(sp), trow + e0, bytes, fb);
          if (need_d) ptx::bulk_g2s(ptx::smem_u32(sp + kHalfSlot), drow + e0, bytes, fb);
        }
        ++task;
        return true;
      };
      while (ok) {
        if (*abort) {
          ok = false;
          break;
        }
        if (rq_c < rq_end) {  // a re-read the control asked for
          const ItemState& it = items[rq_q];
          const int64_t row = ((int64_t)it.b * M + it.n) * V;
          const bool nd = rq_type == kReqRes || it.law.mode == 1;
          ok = issue(rq_type == kReqRes ? kTaskRes : kTaskSearch, rq_q, rq_c, target + row,
                     draft + row, nd);
          ++rq_c;
          t_idle = 0;
          continue;
        }
        int jq = -1;  // a control with a request waiting, taken in turn
        for (int jj = 0; jj < kCtl; ++jj) {
          const int j = (rr + jj) % kCtl;
          if (head[j] < *reinterpret_cast<volatile int*>(&bars->req_tail[j])) {
            jq = j;
            break;
          }
        }
        if (jq >= 0) {
          const int h = head[jq] % kReqQ;
          rq_type = *reinterpret_cast<volatile int*>(&bars->req_type[jq][h]);
          rq_q = *reinterpret_cast<volatile int*>(&bars->req_q[jq][h]);
          const int c = *reinterpret_cast<volatile int*>(&bars->req_c[jq][h]);
          if (rq_type == kReqRes) {
            rq_c = q0;
            rq_end = q1;
          } else {
            rq_c = c;
            rq_end = c + 1;
          }
          ++head[jq];
          rr = (jq + 1) % kCtl;
          t_idle = 0;
          continue;
        }
        if (cur_q >= 0 && s_next < q1) {
          ok = issue(kTaskStats, cur_q, s_next, cur_t, cur_d, cur_pair);
          ++s_next;
          t_idle = 0;
          continue;
        }
        if (!items_done) {
          const int q = k_item % kNQ;
          if (ptx::mbar_test_wait(ptx::smem_u32(&bars->meta[q]), (uint32_t)((k_item / kNQ) & 1))) {
            const ItemState& it = items[q];
            ++k_item;
            *reinterpret_cast<volatile int*>(&bars->prod_items) = k_item;
            t_idle = 0;
            if (it.item < 0) {
              items_done = true;
              cur_q = -1;
            } else {
              cur_q = q;
              s_next = q0;
              cur_pair = it.pair != 0;
              const int64_t row = ((int64_t)it.b * M + it.n) * V;
              cur_t = target + row;
              cur_d = draft + row;
            }
            continue;
          }
        } else if (*reinterpret_cast<volatile int*>(&bars->ctrl_done) == kCtl) {
          break;
        }
        // nothing to issue yet: bounded idle
        const long long now = clock64();
        if (t_idle == 0) {
          t_idle = now;
        } else if ((uint64_t)(now - t_idle) > wait) {
          *abort = 1;
          ok = false;
        }
        if (rq_c >= rq_end) __nanosleep(64);
      }
      if (ok) {
        for (int w = 0; w < kConsumers && ok; ++w) ok = issue(kTaskStop, 0, 0, nullptr, nullptr, false);
      }
      if (!ok) spread_abort();
      // every copy issued lands before the CTA may exit
      for (int64_t u = task > kSlots ? task - kSlots : 0; u < task; ++u)
        ptx::mbar_drain(ptx::smem_u32(&bars->full[u % kSlots]), (uint32_t)((u / kSlots) & 1),
                        kDefaultWaitCycles);
    }
  } else if (warp == kSchedWarp) {
    // ----------------------------------------------------------- scheduler
    // After the last item, one end marker per control (each control takes
    // every kCtl-th slot).
    int stops = 0;
    for (int k = 0;; ++k) {
      const int q = k % kNQ;
      const uint32_t par = (uint32_t)((k / kNQ) & 1);
      if (rank == 0) {
        int i = -1;
        bool ok = true;
        if (lane == 0) {
          // the slot is free once the four controls are done with item k - kNQ
          if (k >= kNQ)
            ok = ptx::mbar_wait_cluster(ptx::smem_u32(&bars->freed[q]), par ^ 1u, abort, wait);
          if (ok) {
            i = (int)atomicAdd(item_counter, 1u);
            if (i >= I) i = -1;
          }
          if (ok && i >= 0) {
            // outputs of a claimed item read -1 until its request is finished
            const int b = i % B, n = i / B;
            out_tokens[(int64_t)b * M + n] = -1;
            path[(int64_t)b * M + n] = -1;
            if (probe != nullptr) store4(probe + ((int64_t)b * M + n) * 4, -1.f, -1.f, -1.f, -1.f);
            if (n == 0) accepted_len[b] = -1;
            __threadfence();
          }
          if (ok) {
            for (uint32_t r = 0; r < kC; ++r) {
              ptx::st_cluster_u32(ptx::map_rank(ptx::smem_u32(&bars->bcast_item[q]), r), (uint32_t)i);
              ptx::mbar_arrive_cluster(ptx::map_rank(ptx::smem_u32(&bars->bcast[q]), r));
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      if (!__all_sync(0xffffffffu, ptx::mbar_wait_cluster(ptx::smem_u32(&bars->bcast[q]), par,
                                                          abort, wait)))
        break;
      ItemState& it = items[q];
      const int i = bars->bcast_item[q];
      if (i < 0) {
        if (lane == 0) {
          it.item = -1;
          ptx::mbar_arrive(ptx::smem_u32(&bars->meta[q]));
        }
        if (++stops == kCtl) break;
        continue;
      }
      const int b = i % B, n = i / B;
      // children of n (ascending), their tokens, the topology check
      uint32_t bad = 0;
      const float temp = temperature[b];
      if (!temperature_valid(temp)) bad |= 1u << SPEC_ERR_INVALID_ARG;
      int pn = n - 1;
      unsigned long long kids = 0;
      if (parent == nullptr) {
        if (n + 1 < M) kids = 1ull;  // bit j: child n + 1 + j
      } else {
        const int32_t* pr = parent + (int64_t)b * M;
        pn = pr[n];
        if (n == 0 ? pn != -1 : (pn < 0 || pn >= n)) bad |= 1u << SPEC_ERR_INVALID_ARG;
        for (int base = n + 1; base < M; base += kWarp) {
          const int c = base + lane;
          const bool is_kid = c < M && pr[c] == n;
          const unsigned bal = __ballot_sync(0xffffffffu, is_kid);
          kids |= (unsigned long long)bal << (base - n - 1);
        }
      }
      // list the children
      const int nk = __popcll(kids);
      if (lane == 0) {
        it.item = i;
        it.b = b;
        it.n = n;
        it.pair = nk > 0;
        it.nkids = nk;
        it.cs = stat_scale(temp);
        it.greedy = temp == 0.f;
        it.par = n == 0 ? -1 : pn;
        it.have = 0;
        it.s_done = 0;
        it.r_done = 0;
      }
      int j = 0;
      unsigned long long kk = kids;
      while (kk) {
        const int bit = __ffsll((long long)kk) - 1;
        kk &= kk - 1;
        if (lane == 0) it.kid[j] = n + 1 + bit;
        ++j;
      }
      __syncwarp();
      for (int jj = lane; jj < nk; jj += kWarp) {
        const int32_t x = tokens[(int64_t)b * M + it.kid[jj]];
        it.ktok[jj] = x;
        if (x < 0 || x >= V) bad |= 1u << SPEC_ERR_DEVICE_BOUNDS;
      }
      bad = __reduce_or_sync(0xffffffffu, bad);
      __syncwarp();
      if (lane == 0) {
        it.bad = bad;
        ptx::mbar_arrive(ptx::smem_u32(&bars->meta[q]));  // releases the state to the CTA
      }
    }
  } else if (warp < kCtrlWarp + kCtl) {
    // ------------------------------------------------------------- control
    const int cj = warp - kCtrlWarp;  // this control's items: k = cj, cj + kCtl, ...
    int e = 0;                  // exchange events of this control so far
    int res_uses[kNQ], srch_uses[kNQ], drawn_uses[kNQ];
    for (int q = 0; q < kNQ; ++q) res_uses[q] = srch_uses[q] = drawn_uses[q] = 0;
    int req_tail = 0;
    bool ok = true;

    // Send `m` (the first `words` 16-byte words of an XMsg) to every CTA
    // of the cluster and wait for theirs: returns the four messages.
    auto exchange = [&](const XMsg& m, int words) -> const XMsg* {
      const int slot = e % kNE;
      XMsg* chan = &xbuf[(cj * kNE + slot) * kC];
      XMsg* dst = &chan[rank];
      const uint4* src = reinterpret_cast<const uint4*>(&m);
      for (int w = lane; w < words * kC; w += kWarp) {
        const int r = w / words, wi = w % words;
        ptx::st_cluster_v4(ptx::map_rank(ptx::smem_u32(reinterpret_cast<uint4*>(dst) + wi), r),
                           src[wi]);
      }
      __syncwarp();
      if (lane == 0) {
        ptx::fence_acq_rel_cluster();
        for (uint32_t r = 0; r < kC; ++r)
          ptx::mbar_arrive_cluster(ptx::map_rank(ptx::smem_u32(&bars->xbar[cj][slot]), r));
      }
      const bool got = __all_sync(0xffffffffu,
                                  ptx::mbar_wait_cluster(ptx::smem_u32(&bars->xbar[cj][slot]),
                                                         (uint32_t)((e / kNE) & 1), abort, wait));
      ++e;
      return got ? chan : nullptr;
    };
    auto request = [&](int type, int q, int c) {
      if (lane == 0) {
        const int h = req_tail % kReqQ;
        bars->req_type[cj][h] = type;
        bars->req_q[cj][h] = q;
        bars->req_c[cj][h] = c;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&bars->req_tail[cj]) = req_tail + 1;
      }
      ++req_tail;
      __syncwarp();
    };
    // A residual pass over the quarter under `L`: its mass, summed over the
    // cluster (rank order).  `qmass` gets the four quarters' masses.
    auto residual_pass = [&](int q, const Law& L, double (&qmass)[kC]) -> bool {
      ItemState& it = items[q];
      if (lane == 0) {
        it.law = L;
        it.r_done = 0;
      }
      __syncwarp();
      double mass = 0.0;
      if (nq > 0) {
        request(kReqRes, q, 0);
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->resd[q]),
                                                    (uint32_t)(res_uses[q] & 1), abort, wait)))
          return false;
        ++res_uses[q];
        for (int j = 0; j < nq; ++j) mass += it.res[j];
      }
      XMsg m;
      m.s_t = mass;
      const XMsg* x = exchange(m, 2);
      if (x == nullptr) return false;
      for (int r = 0; r < kC; ++r) qmass[r] = x[r].s_t;
      return true;
    };

    for (int k = cj; ok; k += kCtl) {
      const int q = k % kNQ;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->meta[q]),
                                                  (uint32_t)((k / kNQ) & 1), abort, wait))) {
        ok = false;
        break;
      }
      ItemState& it = items[q];
      if (it.item < 0) break;
      const int b = it.b, n = it.n, nk = it.nkids;
      const float cs = it.cs;
      // the quarter's statistics
      if (nq > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->stats[q]),
                                                            (uint32_t)((k / kNQ) & 1), abort, wait))) {
        ok = false;
        break;
      }
      // path state of the node from its parent's record (rank 0 reads it,
      // as late as it can, and sends it with its statistics, so all four
      // agree)
      uint32_t pstate = kPathUnknown;
      if (rank == 0 && lane == 0) {
        if (n == 0) {
          pstate = kPathOn;
        } else {
          const Rec* pr = recs + (int64_t)b * M + it.par;
          const uint32_t done = __ldcg(&pr->done);
          if (done == tag) {
            __threadfence();  // the record's fields were written before its tag
            const uint32_t pf = __ldcg(&pr->flags);
            const int acc = __ldcg(&pr->acc_child);
            const uint32_t ps = (pf >> kOnShift) & 3u;
            if (acc != n || ps == kPathOff) pstate = kPathOff;
            else pstate = ps;
          }
        }
      }
      pstate = __shfl_sync(0xffffffffu, pstate, 0);
      XMsg m;
      quarter_stats(it.st_t, nq, cs, &m.m_t, &m.s_t);
      if (it.pair) {
        quarter_stats(it.st_d, nq, cs, &m.m_d, &m.s_d);
      } else {
        m.m_d = -INFINITY;
        m.s_d = 0.0;
      }
      m.have = it.have;
      m.flags = it.bad;
      m.path = pstate;
      m.amax_t = m.amax_d = -1;
      if (it.greedy) {
        // the quarter's first maximum of each row (exact comparisons)
        for (int jj = 0; jj < nq; ++jj)
          if (it.st_t[jj].m == m.m_t) {
            m.amax_t = (q0 + jj) * CH + unpack_index(it.st_t[jj].pad);
            break;
          }
        if (it.pair)
          for (int jj = 0; jj < nq; ++jj)
            if (it.st_d[jj].m == m.m_d) {
              m.amax_d = (q0 + jj) * CH + unpack_index(it.st_d[jj].pad);
              break;
            }
      }
      for (int j = 0; j < nk && j < kMaxKids; ++j) m.gz[j] = it.gz[j];
      const int words = (int)((offsetof(XMsg, gz) + sizeof(float2) * nk + 15) / 16);
      const XMsg* x = exchange(m, words);
      if (x == nullptr) {
        ok = false;
        break;
      }
      // ---- the row normalisers and the checks, identical on every CTA ----
      float mT, mD = 0.f;
      double ST, SD = 1.0;
      row_norm(x, false, cs, &mT, &ST);
      uint32_t bad = x[0].flags | x[1].flags | x[2].flags | x[3].flags;
      if (!norm_ok(mT, ST)) bad |= 1u << SPEC_ERR_NONFINITE;
      if (it.pair) {
        row_norm(x, true, cs, &mD, &SD);
        if (!norm_ok(mD, SD)) bad |= 1u << SPEC_ERR_NONFINITE;
      }
      uint32_t state = x[0].path;
      float xm[kC];   // the quarters' target statistics, kept: the buffer is reused
      double xs[kC];
      for (int r = 0; r < kC; ++r) {
        xm[r] = x[r].m_t;
        xs[r] = x[r].s_t;
      }
      float2 gzk[kMaxKids];
      for (int j = 0; j < nk; ++j) {
        gzk[j] = make_float2(NAN, NAN);
        for (int r = 0; r < kC; ++r)
          if ((x[r].have >> j) & 1ull) gzk[j] = x[r].gz[j];
      }
      const bool decide = bad == 0 && state != kPathOff;
      const bool greedy = it.greedy != 0;
      int amaxT = -1, amaxD = -1;  // greedy: each row's first maximum
      if (greedy) {
        for (int r = 0; r < kC && amaxT < 0; ++r)
          if (x[r].m_t == mT && x[r].amax_t >= 0) amaxT = x[r].amax_t;
        for (int r = 0; r < kC && amaxD < 0; ++r)
          if (x[r].m_d == mD && x[r].amax_d >= 0) amaxD = x[r].amax_d;
      }
      // ---- the tests of the children, in order ---------------------------
      const uint64_t bglob = b_base + (uint64_t)b;
      const double cs64 = (double)cs;
      int acc_child = -1, acc_tok = -1;
      double lc = 0.0, lK = 1.0;   // working target P = max(0, p - lc q) / lK
      double zrep = 1.0;           // mass of the last residual taken (1: P = p)
      float pcs[kMaxKids], qcs[kMaxKids];
      for (int j = 0; j < nk; ++j) pcs[j] = qcs[j] = -1.f;
      bool drawn = false;  // the draw at n was arranged
      if (decide && greedy) {
        // temperature 0: a child is accepted iff its token is the argmax;
        // the draw at n is the argmax (residuals of point masses are that
        // point mass, or empty and back to it)
        for (int j = 0; j < nk; ++j) {
          const bool acc = it.ktok[j] == amaxT;
          pcs[j] = acc ? 1.f : 0.f;
          qcs[j] = it.ktok[j] == amaxD ? 1.f : 0.f;
          if (acc) {
            acc_child = it.kid[j];
            acc_tok = it.ktok[j];
            break;
          }
        }
        drawn = true;
      } else if (decide) {
        const float st_f = (float)ST, sd_f = (float)SD;
        for (int j = 0; j < nk && ok; ++j) {
          const int child = it.kid[j];
          const Philox4 rr = philox4x64_10((uint64_t)child + 1, bglob, offset, 0, seed, 0);
          const float u = u24(rr.w[0]);
          const float zt = gzk[j].x, zd = gzk[j].y;
          bool accept;
          if (parent == nullptr) {
            // one ratio, its exponent in fp64, one fp32 exp2 of the fraction
            const double et = ((double)zt - (double)mT) * cs64;
            const double ed = ((double)zd - (double)mD) * cs64;
            if (ed == -INFINITY) {
              accept = et != -INFINITY;
            } else if (et == -INFINITY) {
              accept = false;
            } else {
              const double ee = et - ed;
              const double ei = rint(ee);
              const float ratio = ldexpf(fast_exp2((float)(ee - ei)), (int)fmax(fmin(ei, 300.0), -300.0)) *
                                  (sd_f / st_f);
              accept = u < ratio;
            }
            pcs[j] = exp2f((float)et) / st_f;
            qcs[j] = exp2f((float)ed) / sd_f;
          } else {
            const double P0 = exp2(((double)zt - (double)mT) * cs64) / ST;
            const double Q = exp2(((double)zd - (double)mD) * cs64) / SD;
            const double P = fmax(P0 - lc * Q, 0.0) / lK;
            accept = (double)u * Q < P;
            pcs[j] = (float)P;
            qcs[j] = (float)Q;
          }
          if (accept) {
            acc_child = child;
            acc_tok = it.ktok[j];
            break;
          }
          // rejected: the next working target needs the mass of
          // max(0, p - (lc + lK) q), a pass over the quarter
          const double nc = lc + lK;
          Law L;
          L.mT = mT;
          L.mD = mD;
          L.invST = (float)(1.0 / ST);
          L.invSD = (float)(1.0 / SD);
          L.cs = cs;
          L.c = (float)nc;
          L.mode = 1;
          L.pad = 0;
          double qm[kC];
          if (!residual_pass(q, L, qm)) {
            ok = false;
            break;
          }
          const double K = qm[0] + qm[1] + qm[2] + qm[3];
          if (K > 0.0) {
            zrep = K / lK;
            lc = nc;
            lK = K;
          } else {  // a residual of zero mass: back to p of the node
            zrep = 1.0;
            lc = 0.0;
            lK = 1.0;
          }
          // the masses of the last pass serve the draw if no sibling follows
          if (j == nk - 1 && K > 0.0) {
            // the draw from max(0, p - lc q): locate the quarter, the chunk
            // and the element; only the CTA holding it searches
            const Philox4 rs = philox4x64_10((uint64_t)n + 1, bglob, offset, 0, seed, 0);
            const double t = (double)u24(rs.w[1]) * K;
            double pre = 0.0;
            int owner = -1, lastpos = -1;
            double last_pre = 0.0;
            for (int r = 0; r < kC; ++r) {
              if (qm[r] > 0.0) {
                lastpos = r;
                last_pre = pre;
                if (owner < 0 && pre + qm[r] > t) owner = r;
              }
              if (owner < 0) pre += qm[r];
            }
            if (owner < 0) {
              owner = lastpos < 0 ? 0 : lastpos;
              pre = last_pre;
            }
            if ((int)rank == owner) {
              const double tq = t - pre;
              double cp = 0.0;
              int sel = -1, lp = -1;
              double lp_pre = 0.0;
              for (int jj = 0; jj < nq; ++jj) {
                const double w = it.res[jj];
                if (w > 0.0) {
                  lp = jj;
                  lp_pre = cp;
                  if (sel < 0 && cp + w > tq) sel = jj;
                }
                if (sel < 0) cp += w;
              }
              if (sel < 0) {
                sel = lp < 0 ? 0 : lp;
                cp = lp_pre;
              }
              const double tr = tq - cp;
              if (lane == 0) {
                it.trel_hi = (float)tr;
                it.trel_lo = (float)(tr - (double)(float)tr);
              }
              __syncwarp();
              request(kReqSearch, q, q0 + sel);
              if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->srch[q]),
                                                          (uint32_t)(srch_uses[q] & 1), abort, wait))) {
                ok = false;
                break;
              }
              ++srch_uses[q];
              if (lane == 0) {
                const uint32_t ra = ptx::map_rank(ptx::smem_u32(&bars->draw[q]), 0);
                ptx::st_cluster_u64(ra, pack_draw(it.s_tok, (float)((double)it.s_w / K)));
                ptx::mbar_arrive_cluster(ptx::map_rank(ptx::smem_u32(&bars->drawn[q]), 0));
              }
            }
            drawn = true;
          }
        }
        if (ok && acc_child < 0 && !drawn) {
          // no child (a leaf or the last node of a chain), or a zero-mass
          // residual after the last child: the draw from p, located from the
          // statistics
          const Philox4 rs = philox4x64_10((uint64_t)n + 1, bglob, offset, 0, seed, 0);
          double qm[kC];
          double Z = 0.0;
          for (int r = 0; r < kC; ++r) {
            qm[r] = (xm[r] == -INFINITY) ? 0.0 : xs[r] * (double)fast_exp2((xm[r] - mT) * cs);
            Z += qm[r];
          }
          const double t = (double)u24(rs.w[1]) * Z;
          double pre = 0.0, last_pre = 0.0;
          int owner = -1, lastpos = -1;
          for (int r = 0; r < kC; ++r) {
            if (qm[r] > 0.0) {
              lastpos = r;
              last_pre = pre;
              if (owner < 0 && pre + qm[r] > t) owner = r;
            }
            if (owner < 0) pre += qm[r];
          }
          if (owner < 0) {
            owner = lastpos < 0 ? 0 : lastpos;
            pre = last_pre;
          }
          zrep = 1.0;
          if ((int)rank == owner) {
            const double tq = t - pre;
            double cp = 0.0, lp_pre = 0.0;
            int sel = -1, lp = -1;
            for (int jj = 0; jj < nq; ++jj) {
              const double w = it.st_t[jj].m == -INFINITY
                                   ? 0.0
                                   : it.st_t[jj].s * (double)fast_exp2((it.st_t[jj].m - mT) * cs);
              if (w > 0.0) {
                lp = jj;
                lp_pre = cp;
                if (sel < 0 && cp + w > tq) sel = jj;
              }
              if (sel < 0) cp += w;
            }
            if (sel < 0) {
              sel = lp < 0 ? 0 : lp;
              cp = lp_pre;
            }
            const double tr = tq - cp;
            if (lane == 0) {
              Law L;
              L.mT = mT;
              L.mD = 0.f;
              L.invST = 0.f;
              L.invSD = 0.f;
              L.cs = cs;
              L.c = 0.f;
              L.mode = 0;
              L.pad = 0;
              it.law = L;
              it.trel_hi = (float)tr;
              it.trel_lo = (float)(tr - (double)(float)tr);
            }
            __syncwarp();
            request(kReqSearch, q, q0 + sel);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->srch[q]),
                                                        (uint32_t)(srch_uses[q] & 1), abort, wait))) {
              ok = false;
            } else {
              ++srch_uses[q];
              if (lane == 0) {
                const uint32_t ra = ptx::map_rank(ptx::smem_u32(&bars->draw[q]), 0);
                ptx::st_cluster_u64(ra, pack_draw(it.s_tok, (float)((double)it.s_w / Z)));
                ptx::mbar_arrive_cluster(ptx::map_rank(ptx::smem_u32(&bars->drawn[q]), 0));
              }
            }
          }
          drawn = true;
        }
      }
      if (!ok) break;
      const bool drew = decide && acc_child < 0;
      // ---- rank 0: the item's record, the children's tests, the request --
      if (rank == 0) {
        DrawMsg dm{-1, -1.f};
        if (drew && greedy) {
          dm = DrawMsg{amaxT, 1.f};
        } else if (drew) {
          if (!__all_sync(0xffffffffu, ptx::mbar_wait_cluster(ptx::smem_u32(&bars->drawn[q]),
                                                              (uint32_t)(drawn_uses[q] & 1), abort,
                                                              wait))) {
            ok = false;
            break;
          }
          ++drawn_uses[q];
          dm = bars->draw[q];
        }
        Rec* rec = recs + (int64_t)b * M;
        for (int j = lane; j < nk; j += kWarp) {
          store_rec_f32(rec + it.kid[j], 6, pcs[j]);
          store_rec_f32(rec + it.kid[j], 7, qcs[j]);
        }
        if (lane == 0) {
          const uint32_t st = bad ? kPathOff : state;
          const uint32_t flags = bad | (st << kOnShift) | (drew ? kDrewBit : 0u) |
                                 ((uint32_t)(it.par + 1) << kParShift);
          Rec* me = rec + n;
          store_rec_u32(me, 1, flags);
          store_rec_u32(me, 2, (uint32_t)acc_child);
          store_rec_u32(me, 3, (uint32_t)(acc_child >= 0 ? acc_tok : dm.tok));
          store_rec_f32(me, 4, drew ? (float)zrep : -1.f);
          store_rec_f32(me, 5, drew ? dm.psamp : -1.f);
          __threadfence();
          store_rec_u32(me, 0, tag);
        }
        __syncwarp();
        __threadfence();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(req_done + b, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (uint32_t)(M - 1)) {
          // ---- every item of request b is finished: its outputs ----------
          __threadfence();
          uint32_t any_bad = 0;
          for (int nn = lane; nn < M; nn += kWarp) any_bad |= __ldcg(&rec[nn].flags) & 0xffu;
          any_bad = __reduce_or_sync(0xffffffffu, any_bad);
          int32_t* ob = out_tokens + (int64_t)b * M;
          int32_t* pb = path + (int64_t)b * M;
          float* prb = probe != nullptr ? probe + (int64_t)b * M * 4 : nullptr;
          if (any_bad) {
            for (int nn = lane; nn < M; nn += kWarp) {
              ob[nn] = -1;
              pb[nn] = -1;
              if (prb) store4(prb + nn * 4, -1.f, -1.f, -1.f, -1.f);
            }
            if (lane == 0) {
              accepted_len[b] = -1;
              raise_status(status, (any_bad >> SPEC_ERR_INVALID_ARG) & 1u ? SPEC_ERR_INVALID_ARG
                                   : (any_bad >> SPEC_ERR_DEVICE_BOUNDS) & 1u ? SPEC_ERR_DEVICE_BOUNDS
                                                                               : SPEC_ERR_NONFINITE);
            }
          } else {
            // walk from the root (one lane), then the rows (all lanes)
            unsigned long long onpath = 0;
            int a = 0, last = 0;
            if (lane == 0) {
              int node = 0;
              onpath = 1ull;
              pb[0] = 0;
              for (int guard = 0; guard < M; ++guard) {
                const int ch = __ldcg(&rec[node].acc_child);
                if (ch < 0 || ch >= M) break;
                ob[a] = __ldcg(&rec[node].tok);
                ++a;
                pb[a] = ch;
                onpath |= 1ull << ch;
                node = ch;
              }
              last = node;
              ob[a] = __ldcg(&rec[node].tok);
              accepted_len[b] = a;
            }
            a = __shfl_sync(0xffffffffu, a, 0);
            last = __shfl_sync(0xffffffffu, last, 0);
            onpath = __shfl_sync(0xffffffffu, onpath, 0);
            for (int nn = lane; nn < M; nn += kWarp) {
              if (nn > a) {
                ob[nn] = -1;
                pb[nn] = -1;
              }
              if (prb) {
                const uint32_t f = __ldcg(&rec[nn].flags);
                const int pp = (int)((f >> kParShift) & 0xffu) - 1;
                float4 v = make_float4(-1.f, -1.f, -1.f, -1.f);
                if (nn > 0 && pp >= 0 && ((onpath >> pp) & 1ull)) {
                  v.x = __ldcg(&rec[nn].pc);
                  v.y = __ldcg(&rec[nn].qc);
                }
                if (nn == last) {
                  v.z = __ldcg(&rec[nn].z);
                  v.w = __ldcg(&rec[nn].psamp);
                }
                store4(prb + nn * 4, v.x, v.y, v.z, v.w);
              }
            }
          }
          if (lane == 0) req_done[b] = 0;  // ready for the next call
        }
      }
      // the slot may be reused once all four controls are done with it and
      // this CTA's producer has taken the item (it reads the state's
      // "next item" only once)
      __syncwarp();
      if (lane == 0) {
        long long t0 = 0;
        while (*reinterpret_cast<volatile int*>(&bars->prod_items) <= k && !*abort) {
          const long long now = clock64();
          if (t0 == 0) t0 = now;
          else if ((uint64_t)(now - t0) > wait) *abort = 1;
        }
        ptx::mbar_arrive_cluster(ptx::map_rank(ptx::smem_u32(&bars->freed[q]), 0));
      }
      __syncwarp();
      if (__shfl_sync(0xffffffffu, *abort, 0)) {
        ok = false;
        break;
      }
    }
    if (lane == 0) atomicAdd(&bars->ctrl_done, 1);
    if (!ok && lane == 0) spread_abort();
  } else {
    // ----------------------------------------------------------- consumers
    const int w = warp - kFirstConsumer;
    for (int64_t t = w;; t += kConsumers) {
      const int slot = (int)(t % kSlots);
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->full[slot]),
                                                  (uint32_t)((t / kSlots) & 1), abort, wait)))
        break;
      const TaskDesc td = bars->task[slot];
      if (td.type == kTaskStop) break;
      ItemState& it = items[td.q];
      const uint8_t* sp = ring + (size_t)slot * kSlotBytes;
      const uint4* sv_t = reinterpret_cast<const uint4*>(sp);
      const uint4* sv_d = reinterpret_cast<const uint4*>(sp + kHalfSlot);
      const int e0 = td.c * CH;
      const int nvalid = V - e0;
      if (td.type == kTaskStats) {
        uint4 raw[kStatVecs];
#pragma unroll
        for (int v = 0; v < kStatVecs; ++v) raw[v] = sv_t[v * kWarp + lane];
        float s_t;
        const float m_t = chunk_stat<T>(raw, nvalid, it.cs, &s_t);
        const bool greedy = it.greedy != 0;
        const int am_t = greedy ? chunk_argmax<T>(raw, nvalid, m_t) : 0;
        float m_d = -INFINITY, s_d = 0.f;
        int am_d = 0;
        if (it.pair) {
#pragma unroll
          for (int v = 0; v < kStatVecs; ++v) raw[v] = sv_d[v * kWarp + lane];
          m_d = chunk_stat<T>(raw, nvalid, it.cs, &s_d);
          if (greedy) am_d = chunk_argmax<T>(raw, nvalid, m_d);
        }
        // the children's logits that fall in this chunk
        for (int j = lane; j < it.nkids; j += kWarp) {
          const int x = it.ktok[j];
          if (x >= e0 && x < e0 + CH && x < V) {
            const T* tt = reinterpret_cast<const T*>(sp);
            const T* dd = reinterpret_cast<const T*>(sp + kHalfSlot);
            it.gz[j] = make_float2(to_f32(tt[x - e0]), to_f32(dd[x - e0]));
            atomicOr(&it.have, 1ull << j);
          }
        }
        __syncwarp();
        if (lane == 0) {
          const int jj = td.c - q0;
          it.st_t[jj].m = m_t;
          it.st_t[jj].pad = pack_index(am_t);
          it.st_t[jj].s = (double)s_t;
          it.st_d[jj].m = m_d;
          it.st_d[jj].pad = pack_index(am_d);
          it.st_d[jj].s = (double)s_d;
          __threadfence_block();
          if (atomicAdd(&it.s_done, 1) == nq - 1) ptx::mbar_arrive(ptx::smem_u32(&bars->stats[td.q]));
        }
      } else if (td.type == kTaskRes) {
        // the order of the elements does not matter for a sum: vector
        // v * 32 + lane, as the statistics read them (no bank conflicts)
        const Law L = it.law;
        float acc = 0.f;
#pragma unroll
        for (int v = 0; v < kStatVecs; ++v) {
          float wv[EPV];
          acc += vec_law<T>(sv_t[v * kWarp + lane], sv_d[v * kWarp + lane],
                            (v * kWarp + lane) * EPV, nvalid, L, wv);
        }
        const dfloat tot = df_warp_sum(df_make(acc));
        if (lane == 0) {
          it.res[td.c - q0] = df_to_d(tot);
          __threadfence_block();
          if (atomicAdd(&it.r_done, 1) == nq - 1) ptx::mbar_arrive(ptx::smem_u32(&bars->resd[td.q]));
        }
      } else {  // search
        const Law L = it.law;
        float wsel;
        const int tok = smem_chunk_draw<T>(sv_t, sv_d, e0, nvalid, L,
                                           dfloat{it.trel_hi, it.trel_lo}, &wsel);
        if (lane == 0) {
          it.s_tok = tok;
          it.s_w = wsel;
          ptx::mbar_arrive(ptx::smem_u32(&bars->srch[td.q]));
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->empty[slot]));
    }
  }

  // ---------------------------------------------------------------- exit
  __syncthreads();
  if (tid == 0 && *abort) {
    raise_status(status, SPEC_ERR_TIMEOUT);
    // items nobody claimed read -1 (a claimed one was set to -1 when claimed)
    const uint32_t first = atomicExch(item_counter, (uint32_t)I);
    for (uint32_t i = first; i < (uint32_t)I; ++i) {
      const int b = (int)(i % (uint32_t)B), n = (int)(i / (uint32_t)B);
      out_tokens[(int64_t)b * M + n] = -1;
      path[(int64_t)b * M + n] = -1;
      if (probe != nullptr) store4(probe + ((int64_t)b * M + n) * 4, -1.f, -1.f, -1.f, -1.f);
      if (n == 0) accepted_len[b] = -1;
    }
  }
  ptx::cluster_sync_all();  // no CTA leaves while another may still write into it
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(ctas_done, 1u) == gridDim.x - 1) {
      // the last CTA out: counters back to zero, the epoch advanced
      *reinterpret_cast<volatile uint32_t*>(item_counter) = 0u;
      *reinterpret_cast<volatile uint32_t*>(ctas_done) = 0u;
      *reinterpret_cast<volatile uint32_t*>(epoch) = tag;
    }
  }
}

}  // namespace rsf

int rsf_max_vocab(int logits_dtype) {
  return rsf::kC * rsf::kMaxQuarter * rs_chunk_elems(logits_dtype);
}

bool rsf_supported(const spec_dims& d, bool aligned) {
  return aligned && d.V <= rsf_max_vocab(d.logits_dtype) && d.M <= rsf::kMaxKids + 1;
}

// The automatic choice takes the fused kernel once every CTA of a cluster
// has a chunk of each row; for shorter rows its per-item exchanges cost more
// than the staged kernels' passes.
bool rsf_preferred(const spec_dims& d, bool aligned) {
  return rsf_supported(d, aligned) && (int64_t)d.V >= (int64_t)rsf::kC * rs_chunk_elems(d.logits_dtype);
}

size_t rsf_smem_bytes() { return rsf::kSmemBytes; }

template <typename T>
static cudaError_t rsf_launch_t(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  using namespace rsf;
  const spec_dims& d = a.d;
  char* ws = static_cast<char*>(a.ws);
  cudaError_t e = cudaFuncSetAttribute(rs_fused_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // one CTA per SM, as many clusters as fit at once (all stay resident: the
  // kernel is persistent and its CTAs wait on one another)
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int cached_dev[2] = {-1, -1}, cached_clusters[2] = {0, 0};
  const int ti = sizeof(T) == 2 ? 0 : 1;
  int nclusters = cached_dev[ti] == dev ? cached_clusters[ti] : 0;
  if (nclusters == 0) {
    cudaLaunchConfig_t qc = {};
    qc.gridDim = dim3(kC * 64);
    qc.blockDim = dim3(kThreads);
    qc.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute ca;
    ca.id = cudaLaunchAttributeClusterDimension;
    ca.val.clusterDim.x = kC;
    ca.val.clusterDim.y = 1;
    ca.val.clusterDim.z = 1;
    qc.attrs = &ca;
    qc.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&nclusters, rs_fused_kernel<T>, &qc);
    if (e != cudaSuccess) return e;
    if (nclusters < 1) return cudaErrorInvalidConfiguration;
    cached_dev[ti] = dev;
    cached_clusters[ti] = nclusters;
  }
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = kC;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kC * nclusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, rs_fused_kernel<T>, static_cast<const T*>(a.target),
                         static_cast<const T*>(a.draft), a.tokens, a.parent, a.temperature, a.seed,
                         a.offset, a.b_base, a.out_tokens, a.path, a.accepted_len, a.probe, d,
                         lay.rs_chunks, reinterpret_cast<Rec*>(ws + lay.rsf_rec_off),
                         reinterpret_cast<uint32_t*>(ws + lay.rsf_req_off),
                         reinterpret_cast<uint32_t*>(ws + lay.rsf_ctl_off),
                         reinterpret_cast<uint32_t*>(ws + lay.status_off));
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaGetLastError();
}

cudaError_t rsf_launch(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  return a.d.logits_dtype == SPEC_BF16 ? rsf_launch_t<__nv_bfloat16>(a, lay, st, launches)
                                       : rsf_launch_t<float>(a, lay, st, launches);
}

}  // namespace specv
