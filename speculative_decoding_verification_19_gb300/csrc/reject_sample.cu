// Accept / reject / resample of speculative decoding on the GPU.
//
// Method (page 1 §2.3, §4.1, §4.3; page 2 §2.1-§2.2; page 3 formal
// definition): p = softmax(target/T), q = softmax(draft/T); draft token x is
// accepted iff u*q(x) < p(x); the walk stops at the first rejection and draws
// the replacement from normalize(max(0, p - q)); a walk that reaches a node
// without children draws the bonus token from p.  Tree: children are tried
// in ascending order, each rejection turns the working target P into
// normalize(max(0, P - q)).  Draws use the inverse CDF in vocabulary order
// (smallest k with C_k > u*Z).
//
// Four kernels, each after the first launched as a programmatic dependent of
// the one before (it starts while its predecessor drains and waits for its
// results in-kernel):
//   rs_rowstats(_bulk)_kernel  every (request, row, 2048-logit chunk):
//                       chunk max m_c and s_c = sum exp2((z - m_c)*log2e/T)
//                       (fp32), over every target row and every draft row
//                       that drafted children.  This is the HBM-streaming
//                       pass: each logit is read once (1-D bulk copies into
//                       shared memory for 16-byte aligned rows).
//   rs_decide_kernel    one CTA per request: row normalisers from the chunk
//                       statistics (fp64); a chain's accept tests all at once
//                       (one thread per draft), a tree's walk in order; a
//                       bonus draw (from p) locates its chunk from the
//                       statistics and searches only that chunk; a residual
//                       draw is left for passes 3 and 4.
//   rs_residual_sums_kernel  one CTA per (2 statistics chunks, request) with a
//                       pending residual: mass of max(0, P - q) per chunk.
//   rs_residual_draw_kernel  one CTA per pending request: picks the chunk
//                       from those masses and searches it element by element.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "philox.cuh"
#include "reject_sample.cuh"
#include "rs_device.cuh"
#include "tc_ptx.cuh"

namespace specv {

constexpr int kRsThreads = 256;   // CTA size of the statistics kernel for unaligned rows
constexpr int kDecThreads = 512;  // decide CTA size
constexpr int kDecWarps = kDecThreads / kWarp;
constexpr int kMaxM = kMaxNodes;
constexpr int kMaxSweeps = 256;

// Statistics chunk: one warp task, 32 lanes x 8 vectors (2048 bf16 / 1024 fp32 logits).
int rs_chunk_elems(int logits_dtype) {
  return kWarp * kStatVecs * (logits_dtype == SPEC_BF16 ? 8 : 4);
}
int rs_max_vocab(int logits_dtype) {
  return kMaxSweeps * kDecThreads * (logits_dtype == SPEC_BF16 ? 8 : 4);
}

// ---------------------------------------------------------------------------
// pass 1: chunk statistics
// ---------------------------------------------------------------------------
// A draft row is read only if its node drafted children (for a tree: some
// parent entry names it).  Warp-uniform.
__device__ __forceinline__ bool row_needed(const int32_t* parent, int M, int b, int which, int n) {
  if (which == 0) return true;
  if (parent == nullptr) return n < M - 1;
  const int lane = threadIdx.x % kWarp;
  const int32_t* par = parent + (int64_t)b * M;
  bool f = false;
  for (int k0 = n + 1; k0 < M; k0 += kWarp) {  // children have larger indices
    const int k = k0 + lane;
    f |= k < M && par[k] == n;
  }
  return __any_sync(0xffffffffu, f);
}

struct StatTask {
  int b, which, n, c;
};
__device__ __forceinline__ StatTask stat_task(int64_t t, int n_chunks, int M) {
  StatTask k;
  k.c = (int)(t % n_chunks);
  const int row = (int)((t / n_chunks) % (2 * M));
  k.b = (int)(t / ((int64_t)n_chunks * 2 * M));
  k.which = row / M;
  k.n = row % M;
  return k;
}

// Next task at or after t (stride nw) whose row is needed, or >= ntask.
__device__ __forceinline__ int64_t next_needed(int64_t t, int64_t nw, int64_t ntask, int n_chunks,
                                               const int32_t* parent, int M) {
  while (t < ntask) {
    const StatTask k = stat_task(t, n_chunks, M);
    if (row_needed(parent, M, k.b, k.which, k.n)) break;
    t += nw;
  }
  return t;
}

// One warp per task (request, row, chunk of 2048 bf16 / 1024 fp32 logits):
// chunk max m_c and s_c = sum exp2((z - m_c) * log2e / T), fp32 terms, fp64
// warp sum.  Persistent grid; each warp loads the next task's logits before
// reducing the current ones, so 2 x 4 KB per warp stay in flight.
template <typename T, bool kAligned>
__global__ void __launch_bounds__(kRsThreads) rs_rowstats_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ parent,
    const float* __restrict__ temperature, spec_dims d, int n_chunks, RowStat* __restrict__ stats) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kChunk = kWarp * kStatVecs * EPV;
  const int lane = threadIdx.x % kWarp;
  const int64_t nw = (int64_t)gridDim.x * (kRsThreads / kWarp);
  const int64_t ntask = (int64_t)d.B * 2 * d.M * n_chunks;
  const int M = d.M, V = d.V;
  pdl_trigger();
  pdl_wait();  // the logits may come from the previous kernel
  int64_t t = next_needed((int64_t)blockIdx.x * (kRsThreads / kWarp) + threadIdx.x / kWarp, nw,
                          ntask, n_chunks, parent, M);

  auto row_ptr = [&](const StatTask& k) {
    return (k.which == 0 ? target : draft) + ((int64_t)k.b * M + k.n) * V;
  };
  // raw 16-byte vectors of a task (aligned rows); vectors past V stay unread
  auto load = [&](int64_t tt, uint4 (&raw)[kStatVecs]) {
    const StatTask k = stat_task(tt, n_chunks, M);
    const T* rp = row_ptr(k);
    const int64_t e0 = (int64_t)k.c * kChunk;
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) {
      const int64_t e = e0 + ((int64_t)v * kWarp + lane) * EPV;
      raw[v] = (e + EPV <= V) ? __ldg(reinterpret_cast<const uint4*>(rp + e)) : make_uint4(0, 0, 0, 0);
    }
  };

  uint4 cur[kStatVecs], nxt[kStatVecs];
  if (kAligned && t < ntask) load(t, cur);
  while (t < ntask) {
    const int64_t t2 = next_needed(t + nw, nw, ntask, n_chunks, parent, M);
    if (kAligned && t2 < ntask) load(t2, nxt);
    const StatTask k = stat_task(t, n_chunks, M);
    const float temp = temperature[k.b];
    const float cs = stat_scale(temp);
    const int64_t e0 = (int64_t)k.c * kChunk;
    float f[kStatVecs][EPV];
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) {
      const int64_t e = e0 + ((int64_t)v * kWarp + lane) * EPV;
      if (kAligned) {
        if (e + EPV <= V) {
          unpack16(cur[v], f[v]);
        } else {
#pragma unroll
          for (int i = 0; i < EPV; ++i) f[v][i] = -INFINITY;
        }
      } else {
        load_vec<T, false>(row_ptr(k), e, V, f[v]);
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v)
#pragma unroll
      for (int i = 0; i < EPV; ++i) m = fmaxf(m, f[v][i]);
    m = warp_max(m);
    float sl = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int v = 0; v < kStatVecs; ++v)
#pragma unroll
        for (int i = 0; i < EPV; ++i) sl += fast_exp2((f[v][i] - m) * cs);
    }
    const double sd = warp_sum((double)sl);
    int am = 0;
    if (temp == 0.f) {  // greedy: the chunk's first maximum
      int best = 0x7fffffff;
#pragma unroll
      for (int v = 0; v < kStatVecs; ++v)
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
          const int er = (v * kWarp + lane) * EPV + i;
          if (e0 + er < V && f[v][i] == m && er < best) best = er;
        }
      am = __reduce_min_sync(0xffffffffu, best);
    }
    if (lane == 0) {
      RowStat r;
      r.m = m;
      r.pad = pack_index(am);
      r.s = sd;
      stats[(((int64_t)k.b * 2 + k.which) * M + k.n) * n_chunks + k.c] = r;
    }
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) cur[v] = nxt[v];
    t = t2;
  }
}

// The same statistics for rows whose starts are 16-byte aligned, fed by 1-D
// bulk copies: each of 16 warps keeps a ring of 3 task slots (4 KB each) in
// shared memory, so about 192 KB per SM is in flight while the warps reduce
// earlier tasks.  One persistent CTA per SM.  Waits are bounded; a time-out
// raises SPEC_ERR_TIMEOUT.
constexpr int kBulkWarps = 16;
constexpr int kBulkRing = 3;
constexpr int kBulkSlot = kWarp * kStatVecs * 16;  // bytes per task
constexpr size_t kBulkSmem = (size_t)kBulkWarps * kBulkRing * kBulkSlot +
                             sizeof(uint64_t) * kBulkWarps * kBulkRing + 64 + 1024;
constexpr size_t kPoolSmem = kBulkSmem + sizeof(int4) * kBulkWarps * kBulkRing;
// A chain's last eighth of tasks is a pool claimed in batches by the warps
// that finish their static range first, so that the stream ends together.
constexpr int kPoolBatch = 4;

// Walks a contiguous range of statistics tasks (request, row, chunk; chunks
// fastest) without divisions, skipping rows that are not read.  For a chain
// the tasks are numbered over the rows that are read (each request's M
// target rows, then its first M-1 draft rows), so that equal ranges are
// equal work; for a tree over all 2M rows, with the unread ones skipped.
struct StatCursor {
  int t, end;           // current flat task and end of the range
  int b, which, n, c;   // decoded position
  int nc, M;
  const int32_t* parent;
  __device__ void start(int t0, int t1, int n_chunks, int M_, const int32_t* par) {
    t = t0;
    end = t1;
    nc = n_chunks;
    M = M_;
    parent = par;
    c = t0 % nc;
    const int rows = par == nullptr ? 2 * M - 1 : 2 * M;  // rows numbered per request
    const int row = (t0 / nc) % rows;
    b = t0 / (nc * rows);
    which = row / M;
    n = row % M;
    skip();
  }
  __device__ bool valid() const { return t < end; }
  // move off rows that are not needed (whole rows at a time)
  __device__ void skip() {
    while (t < end && !row_needed(parent, M, b, which, n)) {
      t += nc - c;
      c = 0;
      next_row();
    }
  }
  __device__ void next_row() {
    if (++n == M || (parent == nullptr && which == 1 && n == M - 1)) {
      n = 0;
      // a chain of one node reads no draft row
      if (++which == 2 || (parent == nullptr && M == 1)) {
        which = 0;
        ++b;
      }
    }
  }
  __device__ void next() {
    ++t;
    if (++c == nc) {
      c = 0;
      next_row();
      skip();
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kBulkWarps * kWarp, 1) rs_rowstats_bulk_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ parent,
    const float* __restrict__ temperature, spec_dims d, int n_chunks, RowStat* __restrict__ stats,
    uint32_t* __restrict__ status) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kChunk = kWarp * kStatVecs * EPV;
  pdl_wait();  // the logits may come from the previous kernel
  // the dependent launches only now, when everything before this kernel has
  // completed: the kernel after it (the chain tail, the tree walk) reads
  // its inputs without waiting for this one
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)kBulkWarps * kBulkRing * kBulkSlot);
  int* abort_flag = reinterpret_cast<int*>(bars + kBulkWarps * kBulkRing);
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kBulkWarps * kBulkRing; ++i) ptx::mbar_init(ptx::smem_u32(&bars[i]), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = abort_flag;
  const uint64_t wait = wait_limit_cycles(d);
  const int M = d.M, V = d.V;
  const int nw = gridDim.x * kBulkWarps;
  const int ntask = d.B * (parent == nullptr ? 2 * M - 1 : 2 * M) * n_chunks;
  const int gw = blockIdx.x * kBulkWarps + warp;
  const int per = (ntask + nw - 1) / nw;
  const int t0 = min(ntask, gw * per), t1 = min(ntask, t0 + per);
  uint8_t* myring = ring + (size_t)warp * kBulkRing * kBulkSlot;
  uint64_t* mybars = bars + warp * kBulkRing;

  auto row_ptr = [&](int b, int which, int n) {
    return (which == 0 ? target : draft) + ((int64_t)b * M + n) * V;
  };
  auto issue = [&](const StatCursor& k, int slot) {
    if (lane == 0) {
      const int64_t e0 = (int64_t)k.c * kChunk;
      const int64_t left = (int64_t)V - e0;
      const uint32_t bytes = (uint32_t)((left < kChunk ? left : kChunk) * sizeof(T));
      const uint32_t bar = ptx::smem_u32(&mybars[slot]);
      ptx::mbar_arrive_expect_tx(bar, bytes);
      ptx::bulk_g2s(ptx::smem_u32(myring + slot * kBulkSlot), row_ptr(k.b, k.which, k.n) + e0,
                    bytes, bar);
    }
  };

  StatCursor cp, ci;  // the task being reduced / the next task to fetch
  cp.start(t0, t1, n_chunks, M, parent);
  ci = cp;
  int issued = 0, done = 0;
  for (int k = 0; k < kBulkRing && ci.valid(); ++k) {
    issue(ci, k);
    ++issued;
    ci.next();
  }
  bool ok = true;
  int cur_b = -1;
  float cs = 1.0f;
  bool greedy = false;
  while (cp.valid()) {
    const int slot = done % kBulkRing;
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&mybars[slot]),
                                                 (uint32_t)((done / kBulkRing) & 1), abort, wait))) {
      ok = false;
      break;
    }
    if (cp.b != cur_b) {
      cur_b = cp.b;
      const float temp = temperature[cur_b];
      cs = stat_scale(temp);
      greedy = temp == 0.f;
    }
    const int e0 = cp.c * kChunk;
    const int nvalid = V - e0;  // elements of this chunk inside the row (may exceed kChunk)
    const uint4* sv = reinterpret_cast<const uint4*>(myring + slot * kBulkSlot);
    uint4 raw[kStatVecs];
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) raw[v] = sv[v * kWarp + lane];
    float sd;
    const float m = chunk_stat<T>(raw, nvalid, cs, &sd);
    const int am = greedy ? chunk_argmax<T>(raw, nvalid, m) : 0;
    if (lane == 0) {
      RowStat r;
      r.m = m;
      r.pad = pack_index(am);
      r.s = (double)sd;
      stats[(((int64_t)cp.b * 2 + cp.which) * M + cp.n) * n_chunks + cp.c] = r;
    }
    ++done;
    __syncwarp();
    if (ci.valid()) {
      // the slot's reads are done before the async proxy refills it
      ptx::fence_proxy_async_smem();
      issue(ci, slot);
      ++issued;
      ci.next();
    }
    cp.next();
  }
  // Copies issued but not consumed (only after a wait gave up) land before
  // the CTA exits: these waits ignore the abort flag and keep the default
  // limit, since the copies complete on their own.
  if (lane == 0)
    for (int u = done; u < issued; ++u)
      ptx::mbar_drain(ptx::smem_u32(&mybars[u % kBulkRing]), (uint32_t)((u / kBulkRing) & 1),
                      kDefaultWaitCycles);
  if (!ok && lane == 0) raise_status(status, SPEC_ERR_TIMEOUT);
}

// The same stream for a chain whose warps have many tasks each: the last
// eighth of the tasks is a pool claimed in batches by the warps that finish
// their balanced static range first, so that the stream ends together.
template <typename T>
__global__ void __launch_bounds__(kBulkWarps * kWarp, 1) rs_rowstats_pool_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ parent,
    const float* __restrict__ temperature, spec_dims d, int n_chunks, RowStat* __restrict__ stats,
    uint32_t* __restrict__ status, uint32_t* pool) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kChunk = kWarp * kStatVecs * EPV;
  pdl_wait();  // the logits may come from the previous kernel
  // the dependent launches only now, when everything before this kernel has
  // completed: the kernel after it (the chain tail, the tree walk) reads
  // its inputs without waiting for this one
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)kBulkWarps * kBulkRing * kBulkSlot);
  int* abort_flag = reinterpret_cast<int*>(bars + kBulkWarps * kBulkRing);
  int4* descs = reinterpret_cast<int4*>(reinterpret_cast<uint8_t*>(abort_flag) + 64);
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kBulkWarps * kBulkRing; ++i) ptx::mbar_init(ptx::smem_u32(&bars[i]), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = abort_flag;
  const uint64_t wait = wait_limit_cycles(d);
  const int M = d.M, V = d.V;
  const int nw = gridDim.x * kBulkWarps;
  const int ntask = d.B * (parent == nullptr ? 2 * M - 1 : 2 * M) * n_chunks;
  const int gw = blockIdx.x * kBulkWarps + warp;
  // balanced static ranges over the first seven eighths; the rest is the pool
  const int pool0 = ntask - ntask / 8;
  const int t0 = (int)((int64_t)gw * pool0 / nw), t1 = (int)((int64_t)(gw + 1) * pool0 / nw);
  uint8_t* myring = ring + (size_t)warp * kBulkRing * kBulkSlot;
  uint64_t* mybars = bars + warp * kBulkRing;
  int4* mydesc = descs + warp * kBulkRing;  // the task in each slot: (b, which, n, chunk)

  auto row_ptr = [&](int b, int which, int n) {
    return (which == 0 ? target : draft) + ((int64_t)b * M + n) * V;
  };
  auto issue = [&](const int4& k, int slot) {
    if (lane == 0) {
      mydesc[slot] = k;
      const int64_t e0 = (int64_t)k.w * kChunk;
      const int64_t left = (int64_t)V - e0;
      const uint32_t bytes = (uint32_t)((left < kChunk ? left : kChunk) * sizeof(T));
      const uint32_t bar = ptx::smem_u32(&mybars[slot]);
      ptx::mbar_arrive_expect_tx(bar, bytes);
      ptx::bulk_g2s(ptx::smem_u32(myring + slot * kBulkSlot), row_ptr(k.x, k.y, k.z) + e0,
                    bytes, bar);
    }
  };
  // the next task to fetch: the static range, then batches from the pool
  StatCursor ci;
  ci.start(t0, t1, n_chunks, M, parent);
  bool pool_left = true;
  auto next_task = [&](int4* out) {
    while (!ci.valid()) {
      if (!pool_left) return false;
      int t = 0;
      if (lane == 0) t = (int)atomicAdd(pool, (uint32_t)kPoolBatch);
      t = pool0 + __shfl_sync(0xffffffffu, t, 0);
      if (t >= ntask) {
        pool_left = false;
        return false;
      }
      ci.start(t, min(ntask, t + kPoolBatch), n_chunks, M, parent);
    }
    *out = make_int4(ci.b, ci.which, ci.n, ci.c);
    ci.next();
    return true;
  };

  int issued = 0, done = 0;
  for (int k = 0; k < kBulkRing; ++k) {
    int4 tk;
    if (!next_task(&tk)) break;
    issue(tk, k);
    ++issued;
  }
  bool ok = true;
  int cur_b = -1;
  float cs = 1.0f;
  bool greedy = false;
  while (done < issued) {
    const int slot = done % kBulkRing;
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&mybars[slot]),
                                                 (uint32_t)((done / kBulkRing) & 1), abort, wait))) {
      ok = false;
      break;
    }
    const int4 cp = mydesc[slot];  // the slot's task: (b, which, n, chunk)
    if (cp.x != cur_b) {
      cur_b = cp.x;
      const float temp = temperature[cur_b];
      cs = stat_scale(temp);
      greedy = temp == 0.f;
    }
    const int e0 = cp.w * kChunk;
    const int nvalid = V - e0;  // elements of this chunk inside the row (may exceed kChunk)
    const uint4* sv = reinterpret_cast<const uint4*>(myring + slot * kBulkSlot);
    uint4 raw[kStatVecs];
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) raw[v] = sv[v * kWarp + lane];
    float sd;
    const float m = chunk_stat<T>(raw, nvalid, cs, &sd);
    const int am = greedy ? chunk_argmax<T>(raw, nvalid, m) : 0;
    if (lane == 0) {
      RowStat r;
      r.m = m;
      r.pad = pack_index(am);
      r.s = (double)sd;
      stats[(((int64_t)cp.x * 2 + cp.y) * M + cp.z) * n_chunks + cp.w] = r;
    }
    ++done;
    __syncwarp();
    int4 tk;
    if (next_task(&tk)) {
      // the slot's reads are done before the async proxy refills it
      ptx::fence_proxy_async_smem();
      issue(tk, slot);
      ++issued;
    }
  }
  // Copies issued but not consumed (only after a wait gave up) land before
  // the CTA exits: these waits ignore the abort flag and keep the default
  // limit, since the copies complete on their own.
  if (lane == 0)
    for (int u = done; u < issued; ++u)
      ptx::mbar_drain(ptx::smem_u32(&mybars[u % kBulkRing]), (uint32_t)((u / kBulkRing) & 1),
                      kDefaultWaitCycles);
  if (!ok && lane == 0) raise_status(status, SPEC_ERR_TIMEOUT);
  // every warp counts itself out; the last one leaves the pool at zero for
  // the next call (no warp claims any more by then)
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(pool + 1, 1u) == (uint32_t)(nw - 1)) {
      pool[0] = 0u;
      pool[1] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// Filtered laws (top-k, top-p): the kept prefix of each row
// ---------------------------------------------------------------------------
// Page 2 §5.1: target and draft must sample by one rule (a nucleus-sampling
// target against a differently sampling draft is its example).  A request
// with a top-k count and / or a top-p mass restricts the law of every row it
// uses -- target and draft alike -- to a prefix of the row's tokens ordered
// by logit, largest first, the smaller index first among equal logits: the
// first k, then the shortest prefix of those whose mass reaches top_p times
// their mass.  The prefix is held as (v, idx): a token is kept iff its logit
// is above v, or equal to v with an index at most idx.
//
// One CTA per row, after the statistics pass (the row maximum m comes from
// the chunk statistics).  The k-th token and the top-p cut are found by a
// most-significant-digit-first radix select over 8-bit digits of an
// order-preserving key of the logit (two digits settle a bf16 value, four an
// fp32 one), each digit one pass over the row building a 256-bin histogram
// of counts and of masses exp2((z - m) cs) in shared memory; the tokens equal
// to the cut's value are then taken in index order (one more pass, in tiles,
// with a block-wide prefix count).  Kept mass K = sum over kept tokens of
// exp2((z - m) cs), so that the restricted law is exp2((z - m) cs) / K.
constexpr int kFiltThreads = 512;
constexpr int kFiltWarps = kFiltThreads / kWarp;

// Order key of a logit: larger logits get smaller keys (ascending key = the
// filter's order of values).
__device__ __forceinline__ uint32_t desc_key(float z) {
  const uint32_t b = __float_as_uint(z);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b ^ 0x80000000u);
  return ~ord;
}

struct FilterSmem {
  uint32_t cnt[256];
  unsigned long long mass[256];  // fixed point: 2^40 per unit of exp2((z - m) cs)
  double red[kFiltWarps];
  int wsum[kFiltWarps];
  uint32_t prefix;   // key digits fixed so far
  uint32_t rem;      // tokens still to take inside the prefix (count select)
  double rem_mass;   // mass still to take inside the prefix (mass select)
  double above;      // mass of the tokens before the prefix
  uint32_t group_n;  // tokens of the final group (inside the kept-k set)
  int found_idx;
  float found_val;
  int running;
};
constexpr double kMassScale = 1099511627776.0;  // 2^40

// Whether token e (logit z, key `key`) is in the kept-k set: key group below
// kkey's, or equal with an index at most kidx (kkey = 0xffffffff, kidx =
// INT_MAX keep everything).
__device__ __forceinline__ bool in_kept(uint32_t key, int64_t e, uint32_t kkey, uint32_t kshift,
                                        int kidx) {
  const uint32_t kg = key >> kshift, kk = kkey >> kshift;
  return kg < kk || (kg == kk && e <= (int64_t)kidx);
}

// One radix digit: the histogram of digit `d` (counts, and with kMass the
// masses) over the tokens whose higher digits equal `prefix` and that lie in
// the kept-k set.  Lanes of a warp that fall in one bin are combined first
// (one shared-memory atomic per bin and warp instruction): the masses as 2^40
// fixed point, summed over the group in two 20-bit halves.
template <typename T, bool kAligned, bool kMass>
__device__ void filter_hist(const T* row, int V, float m, float cs, int d, uint32_t prefix,
                            uint32_t kkey, uint32_t kshift, int kidx, FilterSmem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  for (int i = tid; i < 256; i += kFiltThreads) {
    sh.cnt[i] = 0u;
    sh.mass[i] = 0ull;
  }
  __syncthreads();
  const int sh_d = 8 * d;
  // warp-uniform trip count: every lane takes part in the match / reduce
  for (int64_t e0 = (int64_t)warp * kWarp * EPV; e0 < V; e0 += (int64_t)kFiltThreads * EPV) {
    const int64_t e = e0 + (int64_t)lane * EPV;
    float z[EPV];
    if (e < V) {
      load_vec<T, kAligned>(row, e, V, z);
    } else {
#pragma unroll
      for (int i = 0; i < EPV; ++i) z[i] = -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < EPV; ++i) {
      const uint32_t key = desc_key(z[i]);
      const bool in = e + i < V && (d == 3 || (key >> (sh_d + 8)) == (prefix >> (sh_d + 8))) &&
                      in_kept(key, e + i, kkey, kshift, kidx);
      const uint32_t bin = in ? (key >> sh_d) & 255u : 256u + lane;  // out: a group of one
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      const bool leader = lane == __ffs(peers) - 1;
      if (kMass) {
        const unsigned long long fx =
            in ? (unsigned long long)((double)fast_exp2((z[i] - m) * cs) * kMassScale) : 0ull;
        const unsigned hs = __reduce_add_sync(peers, (unsigned)(fx >> 20));
        const unsigned ls = __reduce_add_sync(peers, (unsigned)(fx & 0xfffffu));
        if (in && leader) atomicAdd(&sh.mass[bin], ((unsigned long long)hs << 20) + ls);
      }
      if (in && leader) atomicAdd(&sh.cnt[bin], (uint32_t)__popc(peers));
    }
  }
  __syncthreads();
}

// Exact (fp64) mass of the kept set: tokens with key group below gkey, or
// equal with an index at most gidx, within the kept-k set.
template <typename T, bool kAligned>
__device__ double filter_kept_mass(const T* row, int V, float m, float cs, uint32_t gkey,
                                   uint32_t gshift, int gidx, uint32_t kkey, uint32_t kshift,
                                   int kidx, FilterSmem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x;
  double acc = 0.0;
  for (int64_t e = (int64_t)tid * EPV; e < V; e += (int64_t)kFiltThreads * EPV) {
    float z[EPV];
    load_vec<T, kAligned>(row, e, V, z);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPV; ++i) {
      const uint32_t key = desc_key(z[i]);
      const bool keep = e + i < V && in_kept(key, e + i, gkey, gshift, gidx) &&
                        in_kept(key, e + i, kkey, kshift, kidx);
      if (keep) s += fast_exp2((z[i] - m) * cs);
    }
    acc += (double)s;
  }
  acc = warp_sum(acc);
  __syncthreads();
  if (tid % kWarp == 0) sh.red[tid / kWarp] = acc;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < kFiltWarps; ++w) t += sh.red[w];
  __syncthreads();
  return t;
}

// The j-th (1-based) token in index order whose key group (key >> gshift)
// equals gkey: its index and logit, into sh.found_idx / sh.found_val.
template <typename T, bool kAligned>
__device__ void filter_nth(const T* row, int V, uint32_t gkey, uint32_t gshift, int j,
                           FilterSmem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kVecs = 4;  // vectors per thread per tile, consecutive
  constexpr int kPer = kVecs * EPV;
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  if (tid == 0) {
    sh.running = 0;
    sh.found_idx = -1;
    sh.found_val = -INFINITY;
  }
  __syncthreads();
  for (int64_t t0 = 0; t0 < V; t0 += (int64_t)kFiltThreads * kPer) {
    const int64_t e0 = t0 + (int64_t)tid * kPer;
    float z[kVecs][EPV];
#pragma unroll
    for (int v = 0; v < kVecs; ++v) {
      if (e0 + v * EPV < V) {
        load_vec<T, kAligned>(row, e0 + v * EPV, V, z[v]);
      } else {
#pragma unroll
        for (int i = 0; i < EPV; ++i) z[v][i] = -INFINITY;
      }
    }
    int c = 0;
#pragma unroll
    for (int v = 0; v < kVecs; ++v)
#pragma unroll
      for (int i = 0; i < EPV; ++i)
        c += (e0 + v * EPV + i < V && (desc_key(z[v][i]) >> gshift) == gkey) ? 1 : 0;
    // block-wide exclusive prefix of the counts, in thread (= index) order
    int incl = c;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == kWarp - 1) sh.wsum[warp] = incl;
    __syncthreads();
    int base = sh.running, total = 0;
    for (int w = 0; w < kFiltWarps; ++w) {
      if (w < warp) base += sh.wsum[w];
      total += sh.wsum[w];
    }
    const int excl = base + incl - c;
    if (c > 0 && excl < j && j <= excl + c) {
      int need = j - excl;
#pragma unroll
      for (int v = 0; v < kVecs; ++v)
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
          const int64_t e = e0 + v * EPV + i;
          if (need > 0 && e < V && (desc_key(z[v][i]) >> gshift) == gkey) {
            if (--need == 0) {
              sh.found_idx = (int)e;
              sh.found_val = z[v][i];
            }
          }
        }
    }
    __syncthreads();
    const bool done = sh.running + total >= j;
    __syncthreads();
    if (tid == 0) sh.running += total;
    if (done) break;
    __syncthreads();
  }
  __syncthreads();
}

template <typename T, bool kAligned>
__global__ void __launch_bounds__(kFiltThreads) rs_filter_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ parent,
    const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
    const float* __restrict__ top_p, spec_dims d, int n_chunks, const RowStat* stats,
    FilterInfo* __restrict__ finfo) {
  __shared__ FilterSmem sh;
  const int M = d.M, V = d.V;
  const int which = blockIdx.x / M, n = blockIdx.x % M, b = blockIdx.y;
  const int tid = threadIdx.x;
  FilterInfo* out = finfo + ((int64_t)b * 2 + which) * M + n;
  pdl_trigger();
  pdl_wait();  // the statistics come from the previous kernel
  const float temp = temperature[b];
  const int k = top_k != nullptr ? top_k[b] : 0;
  const float tp = top_p != nullptr ? top_p[b] : 1.0f;
  const bool use_k = k > 0 && k < V;
  const bool use_p = tp < 1.0f;
  bool needed = which == 0 || row_needed(parent, M, b, which, n);
  needed = __syncthreads_or(needed);
  const bool valid = temperature_ok(temp) && k >= 0 && tp > 0.0f && tp <= 1.0f;
  if (!needed || !valid || !(use_k || use_p)) {
    if (tid == 0) *out = FilterInfo{-INFINITY, 0x7fffffff, 0.0};  // nothing filtered
    return;
  }
  const T* row = (which == 0 ? target : draft) + ((int64_t)b * M + n) * V;
  const float cs = stat_scale(temp);
  // the row maximum from its chunk statistics
  const RowStat* st = stats + (((int64_t)b * 2 + which) * M + n) * n_chunks;
  float mx = -INFINITY;
  for (int c = tid; c < n_chunks; c += kFiltThreads) mx = fmaxf(mx, st[c].m);
  mx = warp_max(mx);
  if (tid % kWarp == 0) sh.red[tid / kWarp] = (double)mx;
  __syncthreads();
  float m = -INFINITY;
  for (int w = 0; w < kFiltWarps; ++w) m = fmaxf(m, (float)sh.red[w]);
  __syncthreads();
  if (!(m > -INFINITY && m < INFINITY)) {  // no distribution: the request fails later
    if (tid == 0) *out = FilterInfo{-INFINITY, 0x7fffffff, 0.0};
    return;
  }
  const int last_d = sizeof(T) == 2 ? 2 : 0;  // a bf16 value is settled by two digits
  const uint32_t gshift = 8u * last_d;

  // ---- top-k: the k-th token of the order ---------------------------------
  uint32_t kkey = 0xffffffffu, kshift = 0;
  int kidx = 0x7fffffff;
  if (use_k) {
    if (tid == 0) {
      sh.prefix = 0u;
      sh.rem = (uint32_t)k;
    }
    __syncthreads();
    for (int dg = 3; dg >= last_d; --dg) {
      filter_hist<T, kAligned, false>(row, V, m, cs, dg, sh.prefix, 0xffffffffu, 0, 0x7fffffff,
                                      sh);
      if (tid == 0) {
        uint32_t cum = 0;
        int bin = 255;
        for (int i = 0; i < 256; ++i) {
          if (cum + sh.cnt[i] >= sh.rem) {
            bin = i;
            break;
          }
          cum += sh.cnt[i];
        }
        sh.rem -= cum;
        sh.prefix |= (uint32_t)bin << (8 * dg);
      }
      __syncthreads();
    }
    const uint32_t pk = sh.prefix;
    filter_nth<T, kAligned>(row, V, pk >> gshift, gshift, (int)sh.rem, sh);
    kkey = pk;
    kshift = gshift;
    kidx = sh.found_idx;
    if (!use_p) {
      const float vk = sh.found_val;
      const double K = filter_kept_mass<T, kAligned>(row, V, m, cs, kkey, kshift, kidx,
                                                     0xffffffffu, 0, 0x7fffffff, sh);
      if (tid == 0) *out = FilterInfo{vk, kidx, K};
      return;
    }
  }

  // ---- top-p: the shortest prefix of the kept-k set reaching top_p of its mass
  if (tid == 0) {
    sh.prefix = 0u;
    sh.above = 0.0;
  }
  __syncthreads();
  for (int dg = 3; dg >= last_d; --dg) {
    filter_hist<T, kAligned, true>(row, V, m, cs, dg, sh.prefix, kkey, kshift, kidx, sh);
    if (tid == 0) {
      if (dg == 3) {  // the first digit sees the whole kept-k set
        double tot = 0.0;
        for (int i = 0; i < 256; ++i) tot += (double)sh.mass[i] / kMassScale;
        sh.rem_mass = (double)tp * tot;
      }
      // the first bin whose running mass reaches what is left to take
      double cum = 0.0;
      int bin = -1, last_nz = 0;
      for (int i = 0; i < 256; ++i) {
        if (sh.cnt[i] == 0u) continue;
        last_nz = i;
        const double mi = (double)sh.mass[i] / kMassScale;
        if (cum + mi >= sh.rem_mass) {
          bin = i;
          break;
        }
        cum += mi;
      }
      if (bin < 0) {  // rounding at the very end: the last non-empty bin
        bin = last_nz;
        cum -= (double)sh.mass[bin] / kMassScale;
      }
      sh.rem_mass -= cum;
      sh.above += cum;
      sh.prefix |= (uint32_t)bin << (8 * dg);
      if (dg == last_d) sh.group_n = sh.cnt[bin];
    }
    __syncthreads();
  }
  // The group of equal logits holding the cut: the smallest count j of its
  // tokens (in index order) whose mass reaches what is left.
  const uint32_t gp = sh.prefix >> gshift;
  filter_nth<T, kAligned>(row, V, gp, gshift, 1, sh);  // its value
  const float vp = sh.found_val;
  const double e = (double)fast_exp2((vp - m) * cs);
  const double jd = e > 0.0 ? ceil(sh.rem_mass / e) : 1.0;
  const int jp = jd < 1.0 ? 1 : (jd > (double)sh.group_n ? (int)sh.group_n : (int)jd);
  __syncthreads();
  if (jp > 1) filter_nth<T, kAligned>(row, V, gp, gshift, jp, sh);
  const int pidx = sh.found_idx;
  const double K = filter_kept_mass<T, kAligned>(row, V, m, cs, sh.prefix, gshift, pidx, kkey,
                                                 kshift, kidx, sh);
  if (tid == 0) *out = FilterInfo{vp, pidx, K};
}

// ---------------------------------------------------------------------------
// pass 2: decisions (and bonus draws); passes 3-4: residual draws
// ---------------------------------------------------------------------------
// Weights of the EPV elements starting at e (elements at or past `lim`
// weigh 0 and are not read).
template <typename T, bool kAligned>
__device__ __forceinline__ float vec_weights(const T* trow, const T* drow, int64_t e, int lim,
                                             const DecideCtx& c, int nrej,
                                             float (&w)[16 / sizeof(T)]) {
  constexpr int EPV = 16 / sizeof(T);
  float zt[EPV], zd[EPV];
  if (e >= lim) {
#pragma unroll
    for (int i = 0; i < EPV; ++i) w[i] = 0.f;
    return 0.f;
  }
  load_vec<T, kAligned>(trow, e, lim, zt);
  if (nrej > 0) {
    load_vec<T, kAligned>(drow, e, lim, zd);
  } else {
#pragma unroll
    for (int i = 0; i < EPV; ++i) zd[i] = 0.f;
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPV; ++i) {
    w[i] = (e + i < lim) ? weight_of(zt[i], zd[i], e + i, c, nrej) : 0.f;
    s += w[i];
  }
  return s;
}

// Block-wide fp64 sum over all threads (every thread gets the result).
__device__ __forceinline__ double block_sum(double v, double* scratch) {
  v = warp_sum(v);
  const int w = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int i = 0; i < kDecWarps; ++i) t += scratch[i];
  return t;
}

// Shared state of the block-wide in-chunk search.
struct DrawScratch {
  double wtot[kDecWarps];
  int claim, last;
  int token;
  float w;
};

// Inverse CDF inside one chunk [e0, e0 + len) (len <= blockDim.x * E):
// every thread takes E consecutive elements starting at e0 + tid*E, sums
// their weights (fp32), the block scans the sums in fp64, and the thread
// whose interval holds `trel` walks its elements in fp64 to the first one
// whose running sum exceeds trel.  The result lands in ds->token / ds->w
// (the weight of the drawn element).  Rounding gaps fall back to the last
// element of positive weight.
template <typename T, bool kAligned>
__device__ void chunk_draw(const T* trow, const T* drow, int64_t e0, int len, int V,
                           const DecideCtx& c, int nrej, double trel, DrawScratch* ds) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int E = 2 * EPV;
  const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
  const int64_t e = e0 + (int64_t)tid * E;
  const int lim = (int)min((int64_t)V, e0 + len);
  float w[E];
  float vsf = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    float wk[EPV];
    vsf += vec_weights<T, kAligned>(trow, drow, e + k * EPV, lim, c, nrej, wk);
#pragma unroll
    for (int i = 0; i < EPV; ++i) w[k * EPV + i] = wk[i];
  }
  const double vs = (double)vsf;
  double incl = vs;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == kWarp - 1) ds->wtot[warp] = incl;
  if (tid == 0) {
    ds->claim = (int)blockDim.x;
    ds->last = -1;
  }
  __syncthreads();
  double wpre = 0.0;
  for (int i = 0; i < warp; ++i) wpre += ds->wtot[i];
  const double excl = wpre + incl - vs;
  if (vs > 0.0) atomicMax(&ds->last, tid);
  if (vs > 0.0 && excl <= trel && trel < excl + vs) atomicMin(&ds->claim, tid);
  __syncthreads();
  int owner = ds->claim;
  if (owner == (int)blockDim.x) owner = ds->last;
  if (owner < 0) owner = 0;
  if (tid == owner) {
    double cum = excl;
    int k = -1, lastpos = -1;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (w[i] > 0.f) lastpos = i;
      cum += (double)w[i];
      if (k < 0 && cum > trel) k = i;
    }
    if (k < 0 || w[k] <= 0.f) k = lastpos;
    if (k < 0) k = 0;
    ds->token = (int)(e + k);
    ds->w = w[k];
  }
  __syncthreads();
}

// The draw from p of `node` (a bonus draw, or the fallback after a residual
// of zero mass): the chunk is located from the pass-1 statistics, then
// searched element by element.  Returns the chunk masses' total Z through
// *zsum.  Called by the whole block.
template <typename T, bool kAligned>
__device__ void draw_from_p(const T* trow, const RowStat* st, int n_chunks, int chunk, int V,
                            const DecideCtx& c, double u, DrawScratch* ds, double* s_trel,
                            int* s_chunk, double* zsum) {
  // warp 0 scans the chunk masses (fp64) 32 at a time and picks the chunk
  if (threadIdx.x < kWarp) {
    const int lane = threadIdx.x;
    double Z = 0.0;
    for (int k = lane; k < n_chunks; k += kWarp) Z += chunk_mass(ld_stat_cg(st + k), c.mT, c.cs);
    Z = warp_sum(Z);
    const double t = u * Z;
    double base = 0.0;
    int sel = -1, lastpos = -1;
    double sel_pre = 0.0;
    for (int k0 = 0; k0 < n_chunks && sel < 0; k0 += kWarp) {
      const int k = k0 + lane;
      const double wk = k < n_chunks ? chunk_mass(ld_stat_cg(st + k), c.mT, c.cs) : 0.0;
      double incl = wk;
#pragma unroll
      for (int o = 1; o < kWarp; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const double excl = base + incl - wk;
      const unsigned hit = __ballot_sync(0xffffffffu, wk > 0.0 && excl + wk > t);
      const unsigned pos = __ballot_sync(0xffffffffu, wk > 0.0);
      if (pos) lastpos = k0 + 31 - __clz(pos);
      if (hit) {
        const int l = __ffs(hit) - 1;
        sel = k0 + l;
        sel_pre = __shfl_sync(0xffffffffu, excl, l);
      }
      base += __shfl_sync(0xffffffffu, incl, kWarp - 1);
    }
    if (sel < 0) {  // rounding at the very top: the last chunk with mass
      sel = lastpos < 0 ? 0 : lastpos;
      double pre = 0.0;
      for (int k = lane; k < sel; k += kWarp) pre += chunk_mass(ld_stat_cg(st + k), c.mT, c.cs);
      sel_pre = warp_sum(pre);
    }
    if (lane == 0) {
      *s_chunk = sel;
      *s_trel = t - sel_pre;
      *zsum = Z;
    }
  }
  __syncthreads();
  chunk_draw<T, kAligned>(trow, trow, (int64_t)(*s_chunk) * chunk, chunk, V, c, 0, *s_trel, ds);
}

// ---- one-warp draw inside a statistics chunk (16-byte aligned rows) ------
// Lane l takes the kStatVecs consecutive 16-byte vectors starting at element
// e0 + l * E of the chunk; the lanes' fp32 weight sums are scanned as
// double-floats, and the owning lane's elements are spread over the warp
// (one 32-bit word per lane) and scanned again.  Same law and rounding-gap
// rule as chunk_draw.
template <typename T, bool kFilt = true>
__device__ __forceinline__ float lane_weights(const T* trow, const T* drow, int64_t e0, int V,
                                              const DecideCtx& c, int nrej,
                                              uint4 (&raw_t)[kStatVecs], uint4 (&raw_d)[kStatVecs]) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int E = kStatVecs * EPV;
  const int lane = threadIdx.x % kWarp;
  const int64_t e = e0 + (int64_t)lane * E;
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v) {
    const bool in = e + (v + 1) * EPV <= V;  // rows are whole 16-byte vectors
    raw_t[v] = in ? __ldg(reinterpret_cast<const uint4*>(trow + e) + v) : make_uint4(0, 0, 0, 0);
    raw_d[v] = (in && nrej > 0) ? __ldg(reinterpret_cast<const uint4*>(drow + e) + v)
                                : make_uint4(0, 0, 0, 0);
  }
  float s = 0.f;
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v) {
    if (e + (v + 1) * EPV > V) continue;
    float zt[EPV], zd[EPV];
    unpack16(raw_t[v], zt);
    unpack16(raw_d[v], zd);
#pragma unroll
    for (int i = 0; i < EPV; ++i) s += weight_sel<kFilt>(zt[i], zd[i], e + v * EPV + i, c, nrej);
  }
  return s;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <typename T, bool kFilt = true>
__device__ int warp_chunk_draw(const T* trow, const T* drow, int64_t e0, int V,
                               const DecideCtx& c, int nrej, dfloat trel, float* w_out) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int E = kStatVecs * EPV;  // elements per lane
  constexpr int EW = 4 / sizeof(T);   // elements per 32-bit word
  const int lane = threadIdx.x % kWarp;
  uint4 raw_t[kStatVecs], raw_d[kStatVecs];
  const float vs = lane_weights<T, kFilt>(trow, drow, e0, V, c, nrej, raw_t, raw_d);
  const dfloat incl = df_warp_scan(df_make(vs));
  const dfloat excl = df_sub(incl, df_make(vs));
  const unsigned hit =
      __ballot_sync(0xffffffffu, vs > 0.f && !df_gt(excl, trel) && df_gt(incl, trel));
  const unsigned pos = __ballot_sync(0xffffffffu, vs > 0.f);
  const int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
  const dfloat r = df_sub(trel, df_shfl(excl, owner));  // position inside the owner's segment
  uint32_t wt = 0, wd = 0;  // lane l takes word l of the owner's segment
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t xt = __shfl_sync(0xffffffffu, word_of(raw_t[v], i), owner);
      const uint32_t xd = __shfl_sync(0xffffffffu, word_of(raw_d[v], i), owner);
      if (lane == v * 4 + i) {
        wt = xt;
        wd = xd;
      }
    }
  const int64_t seg = e0 + (int64_t)owner * E;
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
    const bool in = seg + lane * EW + i < V;
    w[i] = in ? weight_sel<kFilt>(zt, zd, seg + lane * EW + i, c, nrej) : 0.f;
    ls += w[i];
  }
  const dfloat cum = df_warp_scan(df_make(ls));
  const dfloat before = df_sub(cum, df_make(ls));
  const unsigned h2 = __ballot_sync(0xffffffffu, ls > 0.f && df_gt(cum, r));
  const unsigned p2 = __ballot_sync(0xffffffffu, ls > 0.f);
  int k = 0;  // element inside the lane
  if (EW == 2) {
    if (h2) {
      k = (w[0] > 0.f && df_gt(df_add(before, df_make(w[0])), r)) ? 0 : 1;
      if (w[k] <= 0.f) k = 1 - k;
    } else {
      k = w[1] > 0.f ? 1 : 0;  // the last element of positive weight
    }
  }
  const int l2 = h2 ? __ffs(h2) - 1 : (p2 ? 31 - __clz(p2) : 0);
  const int tok = (int)(seg + lane * EW + k);
  const float wk = w[EW == 2 ? (k & 1) : 0];
  *w_out = __shfl_sync(0xffffffffu, wk, l2);
  return __shfl_sync(0xffffffffu, tok, l2);
}

// Picks the chunk holding t from per-chunk masses zs[0..n) (fp64, read
// through L2, or from shared memory with kShared), by one warp: the smallest
// k with a positive mass and an inclusive prefix above t, else the last
// chunk of positive mass.  Returns the chunk; *pre = the masses before it.
template <bool kShared = false>
__device__ __forceinline__ int warp_select_chunk(const double* zs, int n, double t, double* pre) {
  const int lane = threadIdx.x % kWarp;
  double base = 0.0;
  int sel = -1, lastpos = -1;
  double sel_pre = 0.0, last_pre = 0.0;
  for (int k0 = 0; k0 < n && sel < 0; k0 += kWarp) {
    const int k = k0 + lane;
    const double wk = k < n ? (kShared ? zs[k] : __ldcg(zs + k)) : 0.0;
    double incl = wk;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double excl = base + incl - wk;
    const unsigned hit = __ballot_sync(0xffffffffu, wk > 0.0 && excl + wk > t);
    const unsigned pos = __ballot_sync(0xffffffffu, wk > 0.0);
    if (pos) {
      const int l = 31 - __clz(pos);
      lastpos = k0 + l;
      last_pre = __shfl_sync(0xffffffffu, excl, l);
    }
    if (hit) {
      const int l = __ffs(hit) - 1;
      sel = k0 + l;
      sel_pre = __shfl_sync(0xffffffffu, excl, l);
    }
    base += __shfl_sync(0xffffffffu, incl, kWarp - 1);
  }
  if (sel < 0) {  // rounding at the very top: the last chunk with mass
    sel = lastpos < 0 ? 0 : lastpos;
    sel_pre = lastpos < 0 ? 0.0 : last_pre;
  }
  *pre = sel_pre;
  return sel;
}

// The draw from p of `node` by one warp (aligned rows): the statistics
// chunk is located as in draw_from_p (fp64), then searched by
// warp_chunk_draw.  Returns the token; *w its weight, *zsum the total.
template <typename T>
__device__ int warp_draw_from_p(const T* trow, const RowStat* st, int n_chunks, int chunk, int V,
                                const DecideCtx& c, double u, float* w, double* zsum) {
  const int lane = threadIdx.x % kWarp;
  double Z = 0.0;
  for (int k = lane; k < n_chunks; k += kWarp) Z += chunk_mass(ld_stat_cg(st + k), c.mT, c.cs);
  Z = warp_sum(Z);
  const double t = u * Z;
  double base = 0.0;
  int sel = -1, lastpos = -1;
  double sel_pre = 0.0;
  for (int k0 = 0; k0 < n_chunks && sel < 0; k0 += kWarp) {
    const int k = k0 + lane;
    const double wk = k < n_chunks ? chunk_mass(ld_stat_cg(st + k), c.mT, c.cs) : 0.0;
    double incl = wk;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double excl = base + incl - wk;
    const unsigned hit = __ballot_sync(0xffffffffu, wk > 0.0 && excl + wk > t);
    const unsigned pos = __ballot_sync(0xffffffffu, wk > 0.0);
    if (pos) lastpos = k0 + 31 - __clz(pos);
    if (hit) {
      const int l = __ffs(hit) - 1;
      sel = k0 + l;
      sel_pre = __shfl_sync(0xffffffffu, excl, l);
    }
    base += __shfl_sync(0xffffffffu, incl, kWarp - 1);
  }
  if (sel < 0) {  // rounding at the very top: the last chunk with mass
    sel = lastpos < 0 ? 0 : lastpos;
    double pre = 0.0;
    for (int k = lane; k < sel; k += kWarp) pre += chunk_mass(ld_stat_cg(st + k), c.mT, c.cs);
    sel_pre = warp_sum(pre);
  }
  *zsum = Z;
  const double trel = t - sel_pre;
  const float th = (float)trel;
  return warp_chunk_draw<T>(trow, trow, (int64_t)sel * chunk, V, c, 0,
                            dfloat{th, (float)(trel - (double)th)}, w);
}

// Shared state of the decisions of one request (one CTA of kDecThreads).
struct DecideSmem {
  int first_child[kMaxM], next_sib[kMaxM], tok[kMaxM];
  float rowM[2][kMaxM];
  double rowS[2][kMaxM];
  float gzt[kMaxM], gzd[kMaxM];  // logits of each drafted token in its parent's rows
  double px[kMaxM], qx[kMaxM];   // p(x_c), q(x_c) under the parent's rows (fp64)
  double uacc[kMaxM], usmp[kMaxM];
  double red[kDecWarps];
  DecideCtx ctx;
  DrawScratch ds;
  int s_node, s_child, s_accept, s_a, s_chunk;
  double s_trel, s_z;
  int chain_rej[kMaxM];  // chain: the accept test of node n failed
  float chain_p[kMaxM], chain_q[kMaxM];
  int rowA[2][kMaxM];    // greedy: each row's largest logit (smallest index)
  // filtered laws: each row's kept prefix (v, idx) and kept mass K
  float fv[2][kMaxM];
  int fi[2][kMaxM];
  double fK[2][kMaxM];
};

// The decisions of request b from its rows' chunk statistics, by one CTA of
// kDecThreads threads: validation, row normalisers, the accept tests (a
// chain's all at once, a tree walked in order with its residual updates),
// and the draw from p; a draw from a residual is left in draws[b]
// (pending = 1) for the caller.  stats_lost: a statistics wait gave up,
// so the request is failed without being decided.
template <typename T, bool kAligned>
__device__ void decide_request(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parent, const float* __restrict__ temperature, uint64_t seed,
    uint64_t offset, uint64_t b_base, int32_t* __restrict__ out_tokens, int32_t* __restrict__ path,
    int32_t* __restrict__ accepted_len, float* __restrict__ probe, const spec_dims& d, int n_chunks,
    int chunk, const RowStat* stats, DrawState* draws, uint32_t* status, int b, bool stats_lost,
    const int32_t* top_k, const float* top_p, const FilterInfo* finfo, DecideSmem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kSweep = kDecThreads * EPV;
  const int tid = threadIdx.x;
  const int warp = tid / kWarp, lane = tid % kWarp;
  const int M = d.M, V = d.V;

  // defined outputs first
  for (int i = tid; i < M; i += kDecThreads) {
    out_tokens[(int64_t)b * M + i] = -1;
    path[(int64_t)b * M + i] = -1;
  }
  if (probe != nullptr)
    for (int i = tid; i < 4 * M; i += kDecThreads) probe[(int64_t)b * M * 4 + i] = -1.f;
  if (tid == 0) draws[b].pending = 0;

  // ---- validation --------------------------------------------------------
  const float temp = temperature[b];
  const bool greedy = temp == 0.f;
  int bad_arg = !temperature_valid(temp);
  if (top_k != nullptr) bad_arg |= top_k[b] < 0;
  if (top_p != nullptr) {
    const float tp = top_p[b];
    bad_arg |= !(tp > 0.0f && tp <= 1.0f);
  }
  // the filter kernel marks a filtered row with its kept mass K > 0 (every
  // row of a request is filtered alike; target row 0 is always read)
  const bool filtered = finfo != nullptr && !greedy && finfo[(int64_t)b * 2 * M].K > 0.0;
  int bad_tok = 0;
  if (tid < M) {
    const int32_t x = tokens[(int64_t)b * M + tid];
    sh.tok[tid] = x;
    if (tid > 0) bad_tok = (x < 0 || x >= V);
    if (parent != nullptr) {
      const int32_t pn = parent[(int64_t)b * M + tid];
      bad_arg |= (tid == 0) ? (pn != -1) : (pn < 0 || pn >= tid);
    }
  }
  bad_arg = __syncthreads_or(bad_arg);
  bad_tok = __syncthreads_or(bad_tok);
  if (stats_lost) {
    if (tid == 0) {
      accepted_len[b] = -1;
      draws[b].pending = 0;
    }
    return;
  }
  if (tid == 0 && !bad_arg) {
    for (int n = 0; n < M; ++n) sh.first_child[n] = -1;
    for (int n = M - 1; n >= 1; --n) {  // ascending sibling lists
      const int p = parent ? parent[(int64_t)b * M + n] : n - 1;
      sh.next_sib[n] = sh.first_child[p];
      sh.first_child[p] = n;
    }
  }
  if (filtered)
    for (int r = tid; r < 2 * M; r += kDecThreads) {
      const FilterInfo f = finfo[(int64_t)b * 2 * M + r];
      sh.fv[r / M][r % M] = f.v;
      sh.fi[r / M][r % M] = f.idx;
      sh.fK[r / M][r % M] = f.K;
    }
  __syncthreads();
  const float cs = stat_scale(temp);

  // gather the logits every accept test will read, all at once
  if (!bad_arg && !bad_tok && tid >= 1 && tid < M) {
    const int p = parent ? parent[(int64_t)b * M + tid] : tid - 1;
    const int64_t o = ((int64_t)b * M + p) * V + sh.tok[tid];
    sh.gzt[tid] = to_f32(target[o]);
    sh.gzd[tid] = to_f32(draft[o]);
  }
  // ---- row normalisers ---------------------------------------------------
  int bad_row = 0;
  if (!bad_arg) {
    for (int r = warp; r < 2 * M; r += kDecWarps) {
      const int which = r / M, n = r % M;
      if (which == 1 && sh.first_child[n] < 0) continue;
      const RowStat* st = stats + (((int64_t)b * 2 + which) * M + n) * n_chunks;
      // the row's chunk statistics, all loads in flight together
      constexpr int kItems = 16;  // n_chunks <= 512
      float im[kItems];
      double is[kItems];
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int c = lane + j * kWarp;
        if (c < n_chunks) {
          const RowStat x = st[c];
          im[j] = x.m;
          is[j] = x.s;
        } else {
          im[j] = -INFINITY;
          is[j] = 0.0;
        }
      }
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < kItems; ++j) m = fmaxf(m, im[j]);
      m = warp_max(m);
      double s = 0.0;
#pragma unroll
      for (int j = 0; j < kItems; ++j)
        if (im[j] != -INFINITY) s += is[j] * (double)fast_exp2((im[j] - m) * cs);
      s = warp_sum(s);
      if (greedy) {
        // the row's first maximum: the first chunk holding m, then its index
        int c_first = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
          const int c = lane + j * kWarp;
          if (c < n_chunks && im[j] == m && c < c_first) c_first = c;
        }
        c_first = __reduce_min_sync(0xffffffffu, c_first);
        if (lane == 0)
          sh.rowA[which][n] = c_first < n_chunks ? c_first * chunk + unpack_index(st[c_first].pad) : 0;
      }
      if (lane == 0) {
        sh.rowM[which][n] = m;
        sh.rowS[which][n] = s;
      }
      bad_row |= !(m > -INFINITY && m < INFINITY && s > 0.0 && s < INFINITY);
    }
  }
  bad_row = __syncthreads_or(bad_row);
  const uint64_t bglob = b_base + (uint64_t)b;
  const double cs64 = (double)cs;
  if (!(bad_arg || bad_tok || bad_row) && tid < M) {
    // everything the sequential walk needs per node, computed in parallel
    const Philox4 r = philox4x64_10((uint64_t)tid + 1, bglob, offset, 0, seed, 0);
    sh.uacc[tid] = (double)u24(r.w[0]);
    sh.usmp[tid] = (double)u24(r.w[1]);
    if (tid >= 1 && parent == nullptr && !filtered) {
      // chain: every draft's test at once.  The exponent of p(x)/q(x) is
      // formed in fp64 and split into integer and fraction, so that one fp32
      // exp2 gives the ratio to about 3e-7 relative.
      const int p = tid - 1;
      const double et = ((double)sh.gzt[tid] - (double)sh.rowM[0][p]) * cs64;  // log2 unnormalised p(x)
      const double ed = ((double)sh.gzd[tid] - (double)sh.rowM[1][p]) * cs64;  // log2 unnormalised q(x)
      const float st_f = (float)sh.rowS[0][p], sd_f = (float)sh.rowS[1][p];
      bool acc;
      if (ed == -INFINITY) {
        acc = et != -INFINITY;  // q(x) = 0: accepted iff p(x) > 0
      } else if (et == -INFINITY) {
        acc = false;            // p(x) = 0 < u q(x)
      } else {
        const double e = et - ed;
        const double ei = rint(e);
        const float ratio =
            ldexpf(fast_exp2((float)(e - ei)), (int)fmax(fmin(ei, 300.0), -300.0)) * (sd_f / st_f);
        acc = (float)sh.uacc[tid] < ratio;  // u < p(x) / q(x)
      }
      sh.chain_rej[tid] = !acc;
      if (probe != nullptr) {
        sh.chain_p[tid] = exp2f((float)et) / st_f;
        sh.chain_q[tid] = exp2f((float)ed) / sd_f;
      }
    } else if (tid >= 1) {
      const int p = parent ? parent[(int64_t)b * M + tid] : tid - 1;
      if (filtered) {
        // the restricted laws: zero outside the kept prefix, over the kept mass
        const int x = sh.tok[tid];
        const bool kt = kept_at(sh.gzt[tid], x, sh.fv[0][p], sh.fi[0][p]);
        const bool kd = kept_at(sh.gzd[tid], x, sh.fv[1][p], sh.fi[1][p]);
        sh.px[tid] = kt ? exp2(((double)sh.gzt[tid] - (double)sh.rowM[0][p]) * cs64) / sh.fK[0][p]
                        : 0.0;
        sh.qx[tid] = kd ? exp2(((double)sh.gzd[tid] - (double)sh.rowM[1][p]) * cs64) / sh.fK[1][p]
                        : 0.0;
      } else {
        sh.px[tid] = exp2(((double)sh.gzt[tid] - (double)sh.rowM[0][p]) * cs64) / sh.rowS[0][p];
        sh.qx[tid] = exp2(((double)sh.gzd[tid] - (double)sh.rowM[1][p]) * cs64) / sh.rowS[1][p];
      }
    }
  }
  __syncthreads();
  if (bad_arg || bad_tok || bad_row) {
    if (tid == 0) {
      accepted_len[b] = -1;
      raise_status(status, bad_arg ? SPEC_ERR_INVALID_ARG
                           : bad_tok ? SPEC_ERR_DEVICE_BOUNDS
                                     : SPEC_ERR_NONFINITE);
    }
    return;
  }

  if (greedy) {
    // ---- temperature 0: exact match with each row's largest logit -------
    // A child is accepted iff its token is its parent's argmax; the first
    // such child of a node is entered; the token drawn at the last node is
    // its argmax (every residual of point masses is that point mass, or
    // empty, which falls back to it).
    if (tid == 0) {
      int node = 0, a = 0;
      path[(int64_t)b * M] = 0;
      for (;;) {
        int next = -1;
        for (int c = sh.first_child[node]; c >= 0; c = sh.next_sib[c]) {
          const bool acc = sh.tok[c] == sh.rowA[0][node];
          if (probe != nullptr) {
            probe[((int64_t)b * M + c) * 4 + 0] = acc ? 1.f : 0.f;
            probe[((int64_t)b * M + c) * 4 + 1] = sh.tok[c] == sh.rowA[1][node] ? 1.f : 0.f;
          }
          if (acc) {
            next = c;
            break;
          }
        }
        if (next < 0) break;
        out_tokens[(int64_t)b * M + a] = sh.tok[next];
        ++a;
        path[(int64_t)b * M + a] = next;
        node = next;
      }
      out_tokens[(int64_t)b * M + a] = sh.rowA[0][node];
      accepted_len[b] = a;
      if (probe != nullptr) {
        probe[((int64_t)b * M + node) * 4 + 2] = 1.f;
        probe[((int64_t)b * M + node) * 4 + 3] = 1.f;
      }
    }
    return;
  }

  if (parent == nullptr && !filtered) {
    // ---- a chain: the walk stops at the first rejected draft ---------------
    if (tid == 0) {
      int fr = M;
      for (int n = 1; n < M; ++n)
        if (sh.chain_rej[n]) {
          fr = n;
          break;
        }
      sh.s_child = fr;
    }
    __syncthreads();
    const int fr = sh.s_child;              // first rejected node, M if none
    const int a = fr < M ? fr - 1 : M - 1;  // accepted drafts = the draw node
    for (int n = tid; n < M; n += kDecThreads) {
      path[(int64_t)b * M + n] = n <= a ? n : -1;
      if (n < a) out_tokens[(int64_t)b * M + n] = sh.tok[n + 1];
      if (probe != nullptr && n >= 1 && n <= min(fr, M - 1)) {
        probe[((int64_t)b * M + n) * 4 + 0] = sh.chain_p[n];
        probe[((int64_t)b * M + n) * 4 + 1] = sh.chain_q[n];
      }
    }
    if (tid == 0) {
      accepted_len[b] = a;
      ctx_no_filter(sh.ctx);
      sh.ctx.mT = sh.rowM[0][a];
      sh.ctx.invST = (float)(1.0 / sh.rowS[0][a]);
      sh.ctx.cs = cs;
      sh.ctx.nrej = fr < M ? 1 : 0;
      if (fr < M) {
        sh.ctx.mD = sh.rowM[1][a];
        sh.ctx.invSD = (float)(1.0 / sh.rowS[1][a]);
      } else {
        sh.ctx.mD = 0.f;
        sh.ctx.invSD = 0.f;
      }
    }
    __syncthreads();
    const double u = sh.usmp[a];
    if (fr < M) {
      // the residual of node a: its chunk masses need a pass over two rows,
      // spread over the whole GPU by the next kernel
      DrawState& st = draws[b];
      for (int i = tid; i < (int)(sizeof(DecideCtx) / 4); i += kDecThreads)
        reinterpret_cast<uint32_t*>(&st.c)[i] = reinterpret_cast<const uint32_t*>(&sh.ctx)[i];
      if (tid == 0) {
        st.node = a;
        st.a = a;
        st.u = u;
        st.pending = 1;
      }
      return;
    }
    // the bonus token from p of the last node
    const T* trow = target + ((int64_t)b * M + a) * V;
    const RowStat* tst = stats + (((int64_t)b * 2 + 0) * M + a) * n_chunks;
    if (kAligned) {
      if (warp == 0) {
        float w;
        double z;
        const int tk = warp_draw_from_p<T>(trow, tst, n_chunks, chunk, V, sh.ctx, u, &w, &z);
        if (lane == 0) {
          out_tokens[(int64_t)b * M + a] = tk;
          if (probe != nullptr) {
            probe[((int64_t)b * M + a) * 4 + 2] = 1.0f;
            probe[((int64_t)b * M + a) * 4 + 3] = (float)((double)w / z);
          }
        }
      }
      return;
    }
    draw_from_p<T, kAligned>(trow, tst, n_chunks, chunk, V, sh.ctx, u, &sh.ds, &sh.s_trel, &sh.s_chunk, &sh.s_z);
    if (tid == 0) {
      out_tokens[(int64_t)b * M + a] = sh.ds.token;
      if (probe != nullptr) {
        probe[((int64_t)b * M + a) * 4 + 2] = 1.0f;
        probe[((int64_t)b * M + a) * 4 + 3] = (float)((double)sh.ds.w / sh.s_z);
      }
    }
    return;
  }

  // ---- the walk of a tree ------------------------------------------------
  if (tid == 0) {
    sh.s_node = 0;
    sh.s_a = 0;
    path[(int64_t)b * M] = 0;
  }
  for (;;) {
    __syncthreads();
    const int node = sh.s_node;
    const T* trow = target + ((int64_t)b * M + node) * V;
    const T* drow = draft + ((int64_t)b * M + node) * V;
    if (tid == 0) {
      ctx_no_filter(sh.ctx);
      sh.ctx.mT = sh.rowM[0][node];
      sh.ctx.invST = (float)(1.0 / (filtered ? sh.fK[0][node] : sh.rowS[0][node]));
      sh.ctx.cs = cs;
      sh.ctx.nrej = 0;
      if (filtered) {
        sh.ctx.vT = sh.fv[0][node];
        sh.ctx.iT = sh.fi[0][node];
      }
      if (sh.first_child[node] >= 0) {
        sh.ctx.mD = sh.rowM[1][node];
        sh.ctx.invSD = (float)(1.0 / (filtered ? sh.fK[1][node] : sh.rowS[1][node]));
        if (filtered) {
          sh.ctx.vD = sh.fv[1][node];
          sh.ctx.iD = sh.fi[1][node];
        }
      } else {
        sh.ctx.mD = 0.f;
        sh.ctx.invSD = 0.f;
      }
      sh.s_child = sh.first_child[node];
    }
    __syncthreads();
    bool moved = false;
    while (sh.s_child >= 0) {
      const int child = sh.s_child;
      if (tid == 0) {
        // accept test of `child` in fp64
        const double Q = sh.qx[child];
        double P = sh.px[child];
        for (int j = 1; j <= sh.ctx.nrej; ++j) P = fmax(P - Q, 0.0) / sh.ctx.Z[j];
        const double u = sh.uacc[child];
        sh.s_accept = (u * Q < P);
        if (probe != nullptr) {
          probe[((int64_t)b * M + child) * 4 + 0] = (float)P;
          probe[((int64_t)b * M + child) * 4 + 1] = (float)Q;
        }
      }
      __syncthreads();
      if (sh.s_accept) {
        moved = true;
        break;
      }
      if (sh.next_sib[child] >= 0 || filtered) {
        // mass of the next residual, needed by the next sibling's test
        // (trees only: a chain node has a single child); for a filtered law
        // after the last child too, so that a residual of zero mass falls
        // back to the node's law before the draw is posted
        const int nrej_next = sh.ctx.nrej + 1;
        double acc = 0.0;
        // eight sweeps' loads in flight at a time (a row of 32k bf16 logits
        // is eight sweeps: one round trip instead of eight)
        int64_t e = (int64_t)tid * EPV;
        for (; e + 7 * (int64_t)kSweep < V; e += 8 * (int64_t)kSweep) {
          float part[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float w[EPV];
            part[k] = vec_weights<T, kAligned>(trow, drow, e + k * (int64_t)kSweep, V, sh.ctx,
                                               nrej_next, w);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) acc += (double)part[k];  // as the loop below sums
        }
        for (; e < V; e += kSweep) {
          float w[EPV];
          acc += (double)vec_weights<T, kAligned>(trow, drow, e, V, sh.ctx, nrej_next, w);  // lim = V
        }
        const double Z = block_sum(acc, sh.red);
        if (tid == 0) {
          if (Z > 0.0) {
            sh.ctx.nrej = sh.ctx.nrej + 1;
            sh.ctx.invZ[sh.ctx.nrej] = (float)(1.0 / Z);
            sh.ctx.Z[sh.ctx.nrej] = Z;
          } else {
            sh.ctx.nrej = 0;  // zero-mass residual: fall back to p of the node
          }
        }
      } else if (tid == 0) {
        sh.ctx.nrej = sh.ctx.nrej + 1;
      }
      if (tid == 0) sh.s_child = sh.next_sib[child];
      __syncthreads();
    }
    if (moved) {
      if (tid == 0) {
        const int child = sh.s_child;
        const int a = sh.s_a + 1;
        sh.s_a = a;
        path[(int64_t)b * M + a] = child;
        out_tokens[(int64_t)b * M + a - 1] = sh.tok[child];
        sh.s_node = child;
      }
      continue;
    }

    // ---- the draw at `node` ----------------------------------------------
    const double u = sh.usmp[node];
    if (tid == 0) accepted_len[b] = sh.s_a;
    // a filtered law's chunk masses are not in the statistics: every draw of
    // a filtered request (residual or not) goes to the residual kernels
    if (sh.ctx.nrej > 0 || filtered) {
      // residual: its chunk masses need a pass over two rows, spread over
      // the whole GPU by the next kernel
      DrawState& st = draws[b];
      for (int i = tid; i < (int)(sizeof(DecideCtx) / 4); i += kDecThreads)
        reinterpret_cast<uint32_t*>(&st.c)[i] = reinterpret_cast<const uint32_t*>(&sh.ctx)[i];
      if (tid == 0) {
        st.node = node;
        st.a = sh.s_a;
        st.u = u;
        st.pending = 1;
      }
      return;
    }
    const RowStat* tst = stats + (((int64_t)b * 2 + 0) * M + node) * n_chunks;
    if (kAligned) {
      if (warp == 0) {
        float w;
        double z;
        const int tk = warp_draw_from_p<T>(trow, tst, n_chunks, chunk, V, sh.ctx, u, &w, &z);
        if (lane == 0) {
          out_tokens[(int64_t)b * M + sh.s_a] = tk;
          if (probe != nullptr) {
            probe[((int64_t)b * M + node) * 4 + 2] = 1.0f;
            probe[((int64_t)b * M + node) * 4 + 3] = (float)((double)w / z);
          }
        }
      }
      return;
    }
    draw_from_p<T, kAligned>(trow, tst, n_chunks, chunk, V, sh.ctx, u, &sh.ds, &sh.s_trel, &sh.s_chunk, &sh.s_z);
    if (tid == 0) {
      out_tokens[(int64_t)b * M + sh.s_a] = sh.ds.token;
      if (probe != nullptr) {
        probe[((int64_t)b * M + node) * 4 + 2] = 1.0f;
        probe[((int64_t)b * M + node) * 4 + 3] = (float)((double)sh.ds.w / sh.s_z);
      }
    }
    return;
  }
}

template <typename T, bool kAligned>
__global__ void __launch_bounds__(kDecThreads) rs_decide_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parent, const float* __restrict__ temperature, uint64_t seed,
    uint64_t offset, uint64_t b_base, int32_t* __restrict__ out_tokens, int32_t* __restrict__ path,
    int32_t* __restrict__ accepted_len, float* __restrict__ probe, spec_dims d, int n_chunks,
    int chunk, const RowStat* stats, DrawState* __restrict__ draws, uint32_t* status,
    const int32_t* top_k, const float* top_p, const FilterInfo* finfo) {
  __shared__ DecideSmem sh;
  pdl_trigger();
  pdl_wait();  // the statistics (and the filters) come from the previous kernels
  // A wait of the statistics kernel that gave up left some statistics
  // unwritten: then no request of the call is decided on them.
  const bool stats_lost = (ld_volatile_u32(status) >> SPEC_ERR_TIMEOUT) & 1u;
  decide_request<T, kAligned>(target, draft, tokens, parent, temperature, seed, offset, b_base,
                              out_tokens, path, accepted_len, probe, d, n_chunks, chunk, stats,
                              draws, status, blockIdx.x, stats_lost, top_k, top_p, finfo, sh);
}

// Passes 3 and 4: the residual draws.
// Pass 3, one CTA per (kResSpan statistics chunks, request) with a pending
// residual: the mass of max(0, P - q) over each of its chunks, all loads in
// flight together (fp32 within a warp, fp64 across warps).
constexpr int kResThreads = 256;
// statistics chunks per CTA (one 16-byte vector per thread each); small spans
// (many short CTAs) measured faster than long ones at 128 requests x 152k
constexpr int kResSpan = 2;
static_assert(kResThreads * 8 == 2048, "a statistics chunk is kResThreads vectors");

__host__ __device__ __forceinline__ int rs_res_spans(int n_chunks) {
  return (n_chunks + kResSpan - 1) / kResSpan;
}

template <typename T, bool kAligned>
__global__ void __launch_bounds__(kResThreads) rs_residual_sums_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, spec_dims d, int n_chunks,
    int chunk, const DrawState* draws, double* __restrict__ zsum) {
  constexpr int EPV = 16 / sizeof(T);
  const int n_spans = rs_res_spans(n_chunks);
  const int sp = (int)(blockIdx.x % n_spans), b = (int)(blockIdx.x / n_spans), tid = threadIdx.x;
  const int warp = tid / kWarp, lane = tid % kWarp;
  __shared__ DecideCtx ctx;
  __shared__ float s_red[kResThreads / kWarp][kResSpan];
  pdl_trigger();
  pdl_wait();  // the decisions come from the previous kernel
  // the draw state in one round trip: the scalars to registers, the law to
  // shared memory
  const DrawState* dsb = draws + b;
  const int pending = dsb->pending, node = dsb->node;
  for (int i = tid; i < (int)(sizeof(DecideCtx) / 4); i += kResThreads)
    reinterpret_cast<uint32_t*>(&ctx)[i] = reinterpret_cast<const uint32_t*>(&dsb->c)[i];
  if (!pending) return;
  __syncthreads();
  const T* trow = target + ((int64_t)b * d.M + node) * d.V;
  const T* drow = draft + ((int64_t)b * d.M + node) * d.V;
  // thread t takes vector t of each chunk of the span
  float acc[kResSpan];
#pragma unroll
  for (int j = 0; j < kResSpan; ++j) {
    const int k = sp * kResSpan + j;
    float w[EPV];
    acc[j] = k < n_chunks ? vec_weights<T, kAligned>(trow, drow,
                                                     (int64_t)k * chunk + (int64_t)tid * EPV, d.V,
                                                     ctx, ctx.nrej, w)
                          : 0.f;
  }
#pragma unroll
  for (int j = 0; j < kResSpan; ++j) {
    const float sj = warp_sum(acc[j]);
    if (lane == 0) s_red[warp][j] = sj;
  }
  __syncthreads();
  if (tid < kResSpan && sp * kResSpan + tid < n_chunks) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kResThreads / kWarp; ++w) t += (double)s_red[w][tid];
    zsum[(int64_t)b * n_chunks + sp * kResSpan + tid] = t;
  }
}

// Pass 4, one CTA per request with a pending residual: picks the chunk from
// the masses and searches it element by element (one warp for aligned rows).
template <typename T, bool kAligned>
__global__ void __launch_bounds__(kResThreads) rs_residual_draw_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, spec_dims d, int n_chunks,
    int chunk, const RowStat* stats, const DrawState* draws, const double* zsum,
    int32_t* __restrict__ out_tokens, float* __restrict__ probe) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int warp = tid / kWarp, lane = tid % kWarp;
  __shared__ DecideCtx ctx;
  __shared__ DrawScratch ds;
  __shared__ int s_chunk;
  __shared__ double s_trel, s_z;
  pdl_trigger();
  pdl_wait();  // the chunk masses come from the previous kernel
  const DrawState* dsb = draws + b;
  const int pending = dsb->pending, node = dsb->node, a_acc = dsb->a;
  const double u = dsb->u;
  for (int i = tid; i < (int)(sizeof(DecideCtx) / 4); i += kResThreads)
    reinterpret_cast<uint32_t*>(&ctx)[i] = reinterpret_cast<const uint32_t*>(&dsb->c)[i];
  if (!pending) return;
  __syncthreads();
  const int M = d.M;
  const T* trow = target + ((int64_t)b * M + node) * d.V;
  const T* drow = draft + ((int64_t)b * M + node) * d.V;
  const double* zs = zsum + (int64_t)b * n_chunks;
  if (warp == 0) {
    double Z = 0.0;
    for (int k = lane; k < n_chunks; k += kWarp) Z += zs[k];
    Z = warp_sum(Z);
    if (Z > 0.0) {
      double pre;
      const int sel = warp_select_chunk(zs, n_chunks, u * Z, &pre);
      if (kAligned) {
        const double trel = u * Z - pre;
        const float th = (float)trel;
        float w;
        const int tk = warp_chunk_draw<T>(trow, drow, (int64_t)sel * chunk, d.V, ctx, ctx.nrej,
                                          dfloat{th, (float)(trel - (double)th)}, &w);
        if (lane == 0) {
          out_tokens[(int64_t)b * M + a_acc] = tk;
          if (probe != nullptr) {
            // a draw from the node's own (filtered) law reports Z = 1
            probe[((int64_t)b * M + node) * 4 + 2] = ctx.nrej > 0 ? (float)Z : 1.0f;
            probe[((int64_t)b * M + node) * 4 + 3] = (float)((double)w / Z);
          }
        }
      }
      if (lane == 0) {
        s_chunk = sel;
        s_trel = u * Z - pre;
      }
    }
    if (lane == 0) s_z = Z;
  }
  __syncthreads();
  if (s_z > 0.0 && kAligned) return;
  double Zrep;
  if (!(s_z > 0.0)) {
    // a residual of zero mass: draw from p of the node instead
    const RowStat* tst = stats + (((int64_t)b * 2 + 0) * M + node) * n_chunks;
    draw_from_p<T, kAligned>(trow, tst, n_chunks, chunk, d.V, ctx, u, &ds, &s_trel, &s_chunk,
                             &s_z);
    Zrep = 1.0;
  } else {
    chunk_draw<T, kAligned>(trow, drow, (int64_t)s_chunk * chunk, chunk, d.V, ctx, ctx.nrej,
                            s_trel, &ds);
    Zrep = ctx.nrej > 0 ? s_z : 1.0;
  }
  if (tid == 0) {
    out_tokens[(int64_t)b * M + a_acc] = ds.token;
    if (probe != nullptr) {
      probe[((int64_t)b * M + node) * 4 + 2] = (float)Zrep;
      probe[((int64_t)b * M + node) * 4 + 3] = (float)((double)ds.w / s_z);
    }
  }
}

// ---------------------------------------------------------------------------
// The tail of a chain in one kernel: decisions, residual masses and the draw
// ---------------------------------------------------------------------------
// For a chain with 16-byte aligned rows and unfiltered laws, the three
// latency-bound kernels after the statistics pass (decide, residual sums,
// residual draw) are one launch: S CTAs per request ("slices").  Every slice
// forms the request's row normalisers from the chunk statistics and makes
// the same accept decisions (a few loads of data still in L2; no slice waits
// for another).  Slice 0 writes the outputs.  After a rejection at node a,
// slice s computes the residual's mass over its share of the statistics
// chunks of a's two rows (one warp per chunk, every load of a chunk in flight
// at once); the slice that finishes last (a fence and a counter) picks the
// chunk from the masses and the token inside it.  A bonus draw from p needs
// no pass over the row: slice 0 picks the chunk from the statistics.
constexpr int kTailThreads = 256;
constexpr int kTailWarps = kTailThreads / kWarp;

constexpr int kTailStage = 2048;  // chunk statistics of one request held in shared memory

struct TailSmem {
  // the request's chunk statistics (row-major), when they fit: maximum,
  // sum, argmax word
  alignas(16) float st_m[kTailStage];  // (also the residual masses as float2 in the last slice)
  float st_s[kTailStage];
  int st_a[kTailStage];
  float rowM[2][kMaxM];
  float rowS[2][kMaxM];     // row sums (the double-float sum rounded to fp32)
  float rowInv[2][kMaxM];  // 1 / rowS, formed once per row
  int rowA[2][kMaxM];
  int tok[kMaxM];
  float gzt[kMaxM], gzd[kMaxM];
  float pp[kMaxM], qq[kMaxM];
  float usmp[kMaxM];  // the draw's uniform at each node
  int first_rej;
  int last;
  int bad;  // bit 0: argument, bit 1: token, bit 2: row without a distribution
  // the last slice's draw
  dfloat dscan[kTailWarps];
  dfloat trel;
  int sel, zero, hit, lastp, tok_out;
  float w_out, Zf;
};

// Inverse CDF inside statistics chunk [e0, e0 + chunk) of the residual of
// node a, by the whole CTA (the last slice): thread t takes the chunk's
// 16-byte vector t of both rows (every chunk of an aligned row is whole
// vectors, the last one maybe shorter), the threads' sums are scanned in
// double-float, and the thread whose interval holds trel walks its
// elements to the first whose running sum exceeds it; a rounding gap falls
// back to the last element of positive weight.  sh.tok_out / sh.w_out get
// the token and its weight.
template <typename T>
__device__ void tail_block_draw(const T* trow, const T* drow, int64_t e0, int V,
                                const DecideCtx& c, dfloat trel, TailSmem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const int64_t e = e0 + (int64_t)tid * EPV;
  float w[EPV];
  float ts = 0.f;
  if (e < V) {
    const uint4 xt = __ldg(reinterpret_cast<const uint4*>(trow + e));
    const uint4 xd = __ldg(reinterpret_cast<const uint4*>(drow + e));
    float ft[EPV], fd[EPV];
    unpack16(xt, ft);
    unpack16(xd, fd);
#pragma unroll
    for (int i = 0; i < EPV; ++i) {
      w[i] = weight_plain(ft[i], fd[i], c, 1);
      ts += w[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPV; ++i) w[i] = 0.f;
  }
  dfloat incl = df_warp_scan(df_make(ts));
  if (lane == kWarp - 1) sh.dscan[warp] = incl;
  if (tid == 0) {
    sh.hit = 0x7fffffff;
    sh.lastp = -1;
  }
  __syncthreads();
  dfloat base = df_make(0.f);
  for (int k = 0; k < warp; ++k) base = df_add(base, sh.dscan[k]);
  incl = df_add(incl, base);
  const dfloat excl = df_sub(incl, df_make(ts));
  if (ts > 0.f && !df_gt(excl, trel) && df_gt(incl, trel)) atomicMin(&sh.hit, tid);
  if (ts > 0.f) atomicMax(&sh.lastp, tid);
  __syncthreads();
  const bool gap = sh.hit == 0x7fffffff;
  const int owner = gap ? (sh.lastp < 0 ? 0 : sh.lastp) : sh.hit;
  if (tid == owner) {
    dfloat cum = excl;
    int k = -1, klast = -1;
#pragma unroll
    for (int i = 0; i < EPV; ++i) {
      if (w[i] > 0.f) {
        klast = i;
        cum = df_add(cum, df_make(w[i]));
        if (k < 0 && df_gt(cum, trel)) k = i;
      }
    }
    if (k < 0 || gap) k = klast;
    if (k < 0) k = 0;
    sh.tok_out = (int)(e + k);
    sh.w_out = w[k];
  }
  __syncthreads();
}

// Row normaliser (m, S, first argmax) of one row by one warp from its chunk
// statistics, formed as rs_decide_kernel forms it: fp32 maximum, fp64 sum of
// the rescaled chunk sums, the first chunk holding the maximum; every load
// of the row in flight at once (n_chunks <= 512).
__device__ __forceinline__ void tail_row_norm(const RowStat* st, int n_chunks, int chunk, float cs,
                                              float* m_out, double* s_out, int* a_out) {
  const int lane = threadIdx.x % kWarp;
  constexpr int kItems = 16;
  float im[kItems];
  double is[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int c = lane + j * kWarp;
    if (c < n_chunks) {
      const RowStat x = ld_stat_cg(st + c);
      im[j] = x.m;
      is[j] = x.s;
    } else {
      im[j] = -INFINITY;
      is[j] = 0.0;
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kItems; ++j) m = fmaxf(m, im[j]);
  m = warp_max(m);
  double s = 0.0;
#pragma unroll
  for (int j = 0; j < kItems; ++j)
    if (im[j] != -INFINITY) s += is[j] * (double)fast_exp2((im[j] - m) * cs);
  s = warp_sum(s);
  int c_first = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int c = lane + j * kWarp;
    if (c < n_chunks && im[j] == m && c < c_first) c_first = c;
  }
  c_first = __reduce_min_sync(0xffffffffu, c_first);
  *m_out = m;
  *s_out = s;
  *a_out = c_first < n_chunks ? c_first * chunk + unpack_index(ld_stat_cg(st + c_first).pad) : 0;
}

template <typename T>
__global__ void __launch_bounds__(kTailThreads, 2) rs_chain_tail_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const float* __restrict__ temperature, uint64_t seed, uint64_t offset, uint64_t b_base,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ path,
    int32_t* __restrict__ accepted_len, float* __restrict__ probe, spec_dims d, int n_chunks,
    int chunk, const RowStat* stats, double* zsum, uint32_t* done_cnt, uint32_t* status, int S,
    int inputs_ready) {
  __shared__ TailSmem sh;
  const int b = blockIdx.x / S, s = blockIdx.x % S;
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const int M = d.M, V = d.V;
  pdl_trigger();
  // Launched once everything before the statistics kernel has completed
  // (inputs_ready), the kernel reads its inputs before the statistics are
  // done: the tokens, the accept tests' logits and their uniforms; after
  // the LM heads it waits for its predecessor first.
  if (!inputs_ready) pdl_wait();
  int32_t x = 0;
  if (tid < M) x = tokens[(int64_t)b * M + tid];
  const float temp = temperature[b];
  const bool greedy = temp == 0.f;
  const bool tok_bad = tid >= 1 && tid < M && (x < 0 || x >= V);
  // the accept tests' logits: draft n's token in the rows of node n - 1
  float g_t = 0.f, g_d = 0.f, uacc = 0.f, usmp = 0.f;
  if (tid >= 1 && tid < M && !tok_bad) {
    const int64_t o = ((int64_t)b * M + tid - 1) * V + x;
    g_t = to_f32(target[o]);
    g_d = to_f32(draft[o]);
  }
  // node tid's uniforms (counter word 0: tid + 1): the accept test of draft
  // tid and the draw at node tid
  const uint64_t bglob = b_base + (uint64_t)b;
  if (!greedy && tid < M) {
    const Philox4 r = philox4x64_10((uint64_t)tid + 1, bglob, offset, 0, seed, 0);
    uacc = u24(r.w[0]);
    usmp = u24(r.w[1]);
  }
  pdl_wait();  // the statistics come from the previous kernel
  int32_t* ot = out_tokens + (int64_t)b * M;
  int32_t* pt = path + (int64_t)b * M;
  float* pr = probe != nullptr ? probe + (int64_t)b * M * 4 : nullptr;
  auto fail = [&](int code) {  // slice 0: the request's outputs say it failed
    if (s != 0) return;
    for (int i = tid; i < M; i += kTailThreads) {
      ot[i] = -1;
      pt[i] = -1;
    }
    if (pr != nullptr)
      for (int i = tid; i < 4 * M; i += kTailThreads) pr[i] = -1.f;
    if (tid == 0) {
      accepted_len[b] = -1;
      if (code >= 0) raise_status(status, code);
    }
  };
  // a statistics wait that gave up: no decision on what it left unwritten
  if ((ld_volatile_u32(status) >> SPEC_ERR_TIMEOUT) & 1u) {
    fail(-1);
    return;
  }
  const float cs = stat_scale(temp);
  if (tid == 0) sh.bad = temperature_valid(temp) ? 0 : 1;
  if (tid < M) sh.tok[tid] = x;
  __syncthreads();
  if (tok_bad) atomicOr(&sh.bad, 2);
  if (tid < M) {
    sh.gzt[tid] = g_t;
    sh.gzd[tid] = g_d;
    sh.usmp[tid] = usmp;
  }
  // row normalisers: target rows 0..M-1, draft rows 0..M-2, one warp a row;
  // the statistics come in one round of loads through shared memory when
  // they fit
  const int rows = 2 * M - 1;
  const bool staged = rows * n_chunks <= kTailStage;
  if (staged) {
    // the statistics of rows 0..M-1 (target) and M..2M-2 (draft rows
    // 0..M-2) are contiguous per row kind: two runs of items, all loads of a
    // thread issued before any is stored
    const RowStat* tgt_st = stats + ((int64_t)b * 2 + 0) * M * n_chunks;
    const RowStat* dft_st = stats + ((int64_t)b * 2 + 1) * M * n_chunks;
    const int nt = M * n_chunks, items = rows * n_chunks;
    constexpr int kPer = kTailStage / kTailThreads;  // 8
    RowStat x[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = k * kTailThreads + tid;
      if (i < items) x[k] = ld_stat_cg(i < nt ? tgt_st + i : dft_st + (i - nt));
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = k * kTailThreads + tid;
      if (i < items) {
        sh.st_m[i] = x[k].m;
        sh.st_s[i] = (float)x[k].s;  // a chunk sum is an fp32 value
        sh.st_a[i] = unpack_index(x[k].pad);
      }
    }
    __syncthreads();
  }
  for (int r = warp; r < rows; r += kTailWarps) {
    const int which = r < M ? 0 : 1, n = r < M ? r : r - M;
    float m, sm;
    int am;
    if (staged) {
      const float* rm = sh.st_m + r * n_chunks;
      float mx = -INFINITY;
      for (int c = lane; c < n_chunks; c += kWarp) mx = fmaxf(mx, rm[c]);
      m = warp_max(mx);
      // the rescaled chunk sums in double-float (products exact by FMA):
      // fp64 arithmetic is slow on this part
      dfloat acc = df_make(0.f);
      int cf = 0x7fffffff;
      for (int c = lane; c < n_chunks; c += kWarp) {
        if (rm[c] != -INFINITY)
          acc = df_add(acc, df_prod(sh.st_s[r * n_chunks + c], fast_exp2((rm[c] - m) * cs)));
        if (rm[c] == m && c < cf) cf = c;
      }
      acc = df_warp_sum(acc);
      sm = df_to_f(acc);
      cf = __reduce_min_sync(0xffffffffu, cf);
      am = cf < n_chunks ? cf * chunk + sh.st_a[r * n_chunks + cf] : 0;
    } else {
      double sd;
      tail_row_norm(stats + (((int64_t)b * 2 + which) * M + n) * n_chunks, n_chunks, chunk, cs,
                    &m, &sd, &am);
      sm = (float)sd;
    }
    if (lane == 0) {
      sh.rowM[which][n] = m;
      sh.rowS[which][n] = sm;
      sh.rowInv[which][n] = 1.0f / sm;
      sh.rowA[which][n] = am;
      if (!(isfinite(m) && sm > 0.f && isfinite(sm))) atomicOr(&sh.bad, 4);
    }
  }
  __syncthreads();
  const int bad = sh.bad;
  if (bad != 0) {
    fail((bad & 1) ? SPEC_ERR_INVALID_ARG : (bad & 2) ? SPEC_ERR_DEVICE_BOUNDS : SPEC_ERR_NONFINITE);
    return;
  }

  // ---- the accept tests of every draft at once (rs_decide_kernel's chain
  // arithmetic) and the first rejection
  if (tid == 0) sh.first_rej = M;
  __syncthreads();
  if (tid >= 1 && tid < M) {
    const int p = tid - 1;
    bool rej;
    float pp, qq;
    if (greedy) {
      rej = x != sh.rowA[0][p];
      pp = rej ? 0.f : 1.f;
      qq = x == sh.rowA[1][p] ? 1.f : 0.f;
    } else {
      const float zt = sh.gzt[tid], zd = sh.gzd[tid];
      const float st_f = sh.rowS[0][p], sd_f = sh.rowS[1][p];
      const bool t_inf = zt == -INFINITY, d_inf = zd == -INFINITY;
      // the exponents of p(x), q(x) (log2 of the unnormalised terms) and of
      // their ratio in double-float (the differences exact, the products by
      // FMA), split into integer and fraction, so that one fp32 exp2 gives
      // the ratio to about 3e-7 relative
      const dfloat et = df_mul_f(df_two_sum(zt, -sh.rowM[0][p]), cs);
      const dfloat ed = df_mul_f(df_two_sum(zd, -sh.rowM[1][p]), cs);
      bool acc;
      if (d_inf) {
        acc = !t_inf;  // q(x) = 0: accepted iff p(x) > 0
      } else if (t_inf) {
        acc = false;   // p(x) = 0 < u q(x)
      } else {
        const dfloat e = df_sub(et, ed);
        const float ei = rintf(e.hi);
        const float f = (e.hi - ei) + e.lo;
        const float ratio =
            ldexpf(fast_exp2(f), (int)fmaxf(fminf(ei, 300.f), -300.f)) * (sd_f / st_f);
        acc = uacc < ratio;
      }
      rej = !acc;
      pp = t_inf ? 0.f : exp2f(df_to_f(et)) / st_f;
      qq = d_inf ? 0.f : exp2f(df_to_f(ed)) / sd_f;
    }
    sh.pp[tid] = pp;
    sh.qq[tid] = qq;
    if (rej) atomicMin(&sh.first_rej, tid);
  }
  __syncthreads();
  const int fr = sh.first_rej;            // first rejected draft, M if none
  const int a = fr < M ? fr - 1 : M - 1;  // accepted drafts = the node that draws
  if (s == 0) {
    for (int n = tid; n < M; n += kTailThreads) {
      pt[n] = n <= a ? n : -1;
      if (n < a) ot[n] = sh.tok[n + 1];
      else if (n > a) ot[n] = -1;
      if (pr != nullptr) {
        const bool tested = n >= 1 && n <= fr && n < M;
        pr[n * 4 + 0] = tested ? sh.pp[n] : -1.f;
        pr[n * 4 + 1] = tested ? sh.qq[n] : -1.f;
        pr[n * 4 + 2] = -1.f;
        pr[n * 4 + 3] = -1.f;
      }
    }
    if (tid == 0) accepted_len[b] = a;
  }
  if (greedy) {
    if (s == 0 && tid == 0) {
      ot[a] = sh.rowA[0][a];
      if (pr != nullptr) {
        pr[a * 4 + 2] = 1.f;
        pr[a * 4 + 3] = 1.f;
      }
    }
    return;
  }
  DecideCtx c;
  ctx_no_filter(c);
  c.mT = sh.rowM[0][a];
  c.invST = sh.rowInv[0][a];
  c.cs = cs;
  const T* trow = target + ((int64_t)b * M + a) * V;
  // the draw's uniform (counter word 0: node a + 1)
  auto draw_u = [&]() { return (double)sh.usmp[a]; };
  if (fr == M) {
    // every draft accepted: the bonus token from p of node a
    if (s != 0 || warp != 0) return;
    const double u = draw_u();
    c.mD = 0.f;
    c.invSD = 0.f;
    c.nrej = 0;
    float w;
    double z;
    const RowStat* tst = stats + (((int64_t)b * 2 + 0) * M + a) * n_chunks;
    const int tk = warp_draw_from_p<T>(trow, tst, n_chunks, chunk, V, c, u, &w, &z);
    if (lane == 0) {
      ot[a] = tk;
      if (pr != nullptr) {
        pr[a * 4 + 2] = 1.0f;
        pr[a * 4 + 3] = (float)((double)w / z);
      }
    }
    return;
  }
  // a rejection: the residual max(0, p_a - q_a), this slice's chunks
  c.mD = sh.rowM[1][a];
  c.invSD = sh.rowInv[1][a];
  c.nrej = 1;
  const T* drow = draft + ((int64_t)b * M + a) * V;
  double* zs = zsum + (int64_t)b * n_chunks;
  // Each warp's first chunk is fixed (warp w of slice s: chunk s * 8 + w);
  // the rest are claimed one at a time from the request's counter, each
  // warp holding its next claim in flight while it works on the current
  // chunk, so that a slice on a less busy SM takes more of them.
  uint32_t* claim = done_cnt + d.B;
  const int nfixed = S * kTailWarps;
  int cc = s * kTailWarps + warp;
  while (cc < n_chunks) {
    uint32_t nxt = 0;
    if (lane == 0) nxt = atomicAdd(claim + b, 1u);
    uint4 raw_t[kStatVecs], raw_d[kStatVecs];
    const float ls = lane_weights<T, false>(trow, drow, (int64_t)cc * chunk, V, c, 1, raw_t, raw_d);
    const dfloat tot = df_warp_sum(df_make(ls));
    if (lane == 0) {
      reinterpret_cast<float2*>(zs)[cc] = make_float2(tot.hi, tot.lo);
      __threadfence();  // the mass before this slice's count
    }
    cc = nfixed + __shfl_sync(0xffffffffu, (int)nxt, 0);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sh.last = atomicAdd(done_cnt + b, 1u) == (uint32_t)(S - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  // the last slice: the chunk from the masses (all loaded at once into
  // shared memory when they fit), then the token
  __threadfence();
  // the masses (double-floats) one chunk a lane, scanned in order by warp
  // 0: the first chunk of positive mass whose running mass exceeds u * Z,
  // else the last of positive mass; then the whole CTA searches that chunk
  const double u = warp == 0 ? draw_u() : 0.0;
  if (warp == 0) {
    // the masses in one round of loads, kept in shared memory (the
    // statistics staging area, free by now) for the scan
    const float2* zf = reinterpret_cast<const float2*>(zs);
    float2* zm = reinterpret_cast<float2*>(sh.st_m);  // 1024 entries >= n_chunks
    dfloat Zd = df_make(0.f);
    for (int k = lane; k < n_chunks; k += kWarp) {
      const float2 v = __ldcg(zf + k);
      zm[k] = v;
      Zd = df_add(Zd, dfloat{v.x, v.y});
    }
    Zd = df_warp_sum(Zd);
    if (Zd.hi > 0.f) {
      const dfloat t = df_mul_f(Zd, (float)u);  // u is a 24-bit fraction: exact in fp32
      dfloat base = df_make(0.f), sel_pre = df_make(0.f), last_pre = df_make(0.f);
      int sel = -1, lastpos = -1;
      for (int k0 = 0; k0 < n_chunks && sel < 0; k0 += kWarp) {
        const int k = k0 + lane;
        const float2 v = k < n_chunks ? zm[k] : make_float2(0.f, 0.f);
        const dfloat wk{v.x, v.y};
        const dfloat incl = df_add(base, df_warp_scan(wk));
        const dfloat excl = df_sub(incl, wk);
        const bool pos = wk.hi > 0.f;
        const unsigned hit = __ballot_sync(0xffffffffu, pos && df_gt(incl, t));
        const unsigned pb = __ballot_sync(0xffffffffu, pos);
        if (pb) {
          const int l = 31 - __clz(pb);
          lastpos = k0 + l;
          last_pre = df_shfl(excl, l);
        }
        if (hit) {
          const int l = __ffs(hit) - 1;
          sel = k0 + l;
          sel_pre = df_shfl(excl, l);
        }
        base = df_shfl(incl, kWarp - 1);
      }
      if (sel < 0) {  // rounding at the very top: the last chunk with mass
        sel = lastpos < 0 ? 0 : lastpos;
        sel_pre = lastpos < 0 ? df_make(0.f) : last_pre;
      }
      if (lane == 0) {
        sh.zero = 0;
        sh.sel = sel;
        sh.trel = df_sub(t, sel_pre);
        sh.Zf = df_to_f(Zd);
      }
    } else if (lane == 0) {
      sh.zero = 1;
    }
  }
  __syncthreads();
  if (!sh.zero) {
    tail_block_draw<T>(trow, drow, (int64_t)sh.sel * chunk, V, c, sh.trel, sh);
    if (tid == 0) {
      ot[a] = sh.tok_out;
      if (pr != nullptr) {
        pr[a * 4 + 2] = sh.Zf;
        pr[a * 4 + 3] = sh.w_out / sh.Zf;
      }
      done_cnt[b] = 0u;  // ready for the next call
      claim[b] = 0u;
    }
    return;
  }
  // a residual of zero mass: the draw from p of the node
  if (warp != 0) return;
  c.nrej = 0;
  float w;
  double z;
  const RowStat* tst = stats + (((int64_t)b * 2 + 0) * M + a) * n_chunks;
  const int tk = warp_draw_from_p<T>(trow, tst, n_chunks, chunk, V, c, u, &w, &z);
  if (lane == 0) {
    ot[a] = tk;
    if (pr != nullptr) {
      pr[a * 4 + 2] = 1.f;
      pr[a * 4 + 3] = (float)((double)w / z);
    }
    done_cnt[b] = 0u;  // ready for the next call
    claim[b] = 0u;
  }
}

// ---------------------------------------------------------------------------
// One kernel for a chain: statistics, decisions and draws, all warps alike.
//
// Every warp streams statistics chunks through a private ring of 4 KB
// shared-memory slots filled by 1-D bulk copies (as rs_rowstats_bulk_kernel
// does), claiming batches of chunks from a global counter in request-major
// order, so that requests are finished one after another while the stream
// goes on.  What the finished chunks make ready is done by the warp that
// makes it ready, between batches, while its next copies are in flight:
//   * the chunks that complete a row: the row's normaliser (max m, sum S in
//     fp64, and its first largest logit) from the row's chunk statistics;
//   * the row that completes a request: the request's decisions (the accept
//     tests of the chain, the number accepted) and, when every draft was
//     accepted, the bonus draw from p; a rejection posts the request's
//     residual chunks (one unit per statistics chunk) to a global list;
//   * a residual unit, claimed from that list by a warp between batches
//     (warps 0..3 of each CTA) or once its stream is over (every warp): the
//     masses of max(0, p - q) over four statistics chunks of the node's rows
//     (re-read while still in L2); the unit that completes a request picks
//     the chunk from the masses and the token inside it.
// Only the decisions of the last requests, and their residual units (spread
// over every warp), come after the stream ends.  A warp's count of finished
// chunks is added to its row's counter at the end of each batch and the
// returned count looked at one batch later, so that the stream never waits
// for the atomic.
//
// Global control words ctl[] (two 128-byte lines: the batch counter, hit
// by every claim, apart from the words idle warps poll):
//   [0] next batch of statistics chunks  [1] residual entries allocated
//   [2] CTAs finished
//   [32] residual units published        [33] residual units claimed
//   [34] requests finished               [35] the call failed (a wait gave up)
// Every counter is back at zero when the call ends (the last CTA out resets
// ctl and the entries' flags; each per-row and per-request counter is reset
// by the warp that saw it complete), so the next call starts clean.  After a
// wait gave up (SPEC_ERR_TIMEOUT) they are not: the workspace is initialised
// again before the next call.
// ---------------------------------------------------------------------------
constexpr int kFWarps = 16;   // warps per CTA (one CTA per SM)
constexpr int kFRing = 3;     // 4 KB slots per warp
constexpr int kFBatch = 4;    // statistics chunks per claim
constexpr int kFUnit = 4;     // statistics chunks per residual unit
constexpr size_t kFSmem = (size_t)kFWarps * kFRing * kBulkSlot + 1024;
constexpr int kFCtl = 64;
constexpr int kCBatch = 0, kCEntries = 1, kCCtas = 2;
constexpr int kCPub = 32, kCClaim = 33, kCFin = 34, kCFail = 35;

// Normaliser of one logits row: its maximum m, S = sum exp2((z - m) cs) and
// the index of its first largest logit.
struct RowNorm {
  float m;
  int amax;
  double S;
};

// A posted residual draw: the request, its node and law, and the uniform;
// `ready` is written last (release) and read first (acquire).
struct ResEntry {
  int b, node, a, pad0;
  float mT, mD, invST, invSD;
  float cs;
  uint32_t ready;
  double u;
};
static_assert(sizeof(ResEntry) == 48, "three 16-byte loads");

struct FusedWs {
  RowStat* stats;
  RowNorm* norms;       // [B][2M]: target row n at n, draft row n at M + n
  uint32_t* row_cnt;    // [B][2M]: statistics chunks finished per row
  uint32_t* req_rows;   // [B]: rows finished per request
  ResEntry* entries;    // [B]: residual draws in the order posted
  uint32_t* res_cnt;    // [B]: residual units finished per request
  double* zsum;         // [B][n_chunks]: residual mass per chunk
  uint32_t* ctl;        // [kFCtl]
  uint32_t* status;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// A chunk statistic written by another SM during this kernel, read through L2.
__device__ __forceinline__ RowStat ld_stat(const RowStat* p) {
  const uint4 r = __ldcg(reinterpret_cast<const uint4*>(p));
  RowStat s;
  s.m = __uint_as_float(r.x);
  s.pad = __uint_as_float(r.y);
  s.s = __hiloint2double((int)r.w, (int)r.z);
  return s;
}

__device__ __forceinline__ RowNorm ld_norm(const RowNorm* p) {
  const uint4 r = __ldcg(reinterpret_cast<const uint4*>(p));
  RowNorm n;
  n.m = __uint_as_float(r.x);
  n.amax = (int)r.y;
  n.S = __hiloint2double((int)r.w, (int)r.z);
  return n;
}

// The normaliser of one row from its chunk statistics (one warp), formed as
// rs_decide_kernel forms it: the fp32 maximum, the fp64 sum of the rescaled
// chunk sums, and the first chunk holding the maximum for the argmax.
__device__ __noinline__ void fused_row_norm(const RowStat* st, int n_chunks, int chunk, float cs,
                                            RowNorm* out) {
  const int lane = threadIdx.x % kWarp;
  constexpr int kItems = 16;  // n_chunks <= 512
  float im[kItems];
  double is[kItems];
  int ia[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int c = lane + j * kWarp;
    if (c < n_chunks) {
      const RowStat x = ld_stat(st + c);
      im[j] = x.m;
      is[j] = x.s;
      ia[j] = unpack_index(x.pad);
    } else {
      im[j] = -INFINITY;
      is[j] = 0.0;
      ia[j] = 0;
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kItems; ++j) m = fmaxf(m, im[j]);
  m = warp_max(m);
  double s = 0.0;
#pragma unroll
  for (int j = 0; j < kItems; ++j)
    if (im[j] != -INFINITY) s += is[j] * (double)fast_exp2((im[j] - m) * cs);
  s = warp_sum(s);
  int c_first = 0x7fffffff, a_first = 0;
#pragma unroll
  for (int j = kItems - 1; j >= 0; --j) {  // this lane's first chunk holding m
    const int c = lane + j * kWarp;
    if (c < n_chunks && im[j] == m) {
      c_first = c;
      a_first = ia[j];
    }
  }
  const int cmin = __reduce_min_sync(0xffffffffu, c_first);
  const unsigned own = __ballot_sync(0xffffffffu, c_first == cmin);
  const int am = __shfl_sync(0xffffffffu, a_first, __ffs(own) - 1);
  if (lane == 0) {
    RowNorm r;
    r.m = m;
    r.amax = cmin < n_chunks ? cmin * chunk + am : 0;
    r.S = s;
    *out = r;
  }
}

// Marks request b finished (its outputs are written).
__device__ __forceinline__ void fused_finish(uint32_t* ctl) {
  if (threadIdx.x % kWarp == 0) {
    __threadfence();
    atomicAdd(ctl + kCFin, 1u);
  }
}

// The decisions of chain request b, by one warp, once every row's normaliser
// is written: validation, the accept tests of every draft at once (the same
// arithmetic as rs_decide_kernel's chain path), the outputs, and the draw
// (bonus from p here; a residual is posted as units).
template <typename T>
__device__ __noinline__ void fused_decide(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const float* __restrict__ temperature, uint64_t seed, uint64_t offset, uint64_t b_base,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ path, int32_t* __restrict__ accepted_len,
    float* __restrict__ probe, const spec_dims& d, int n_chunks, int chunk, const FusedWs& w,
    int b) {
  const int lane = threadIdx.x % kWarp;
  const int M = d.M, V = d.V;
  const float temp = temperature[b];
  const bool greedy = temp == 0.f;
  const float cs = stat_scale(temp);
  const RowNorm* nb = w.norms + (int64_t)b * 2 * M;
  int32_t* ot = out_tokens + (int64_t)b * M;
  int32_t* pt = path + (int64_t)b * M;
  float* pr = probe != nullptr ? probe + (int64_t)b * M * 4 : nullptr;

  // validation: the temperature, the drafted tokens, every row's normaliser
  bool bad_arg = !temperature_valid(temp), bad_tok = false, bad_row = false;
  for (int n = lane; n < M; n += kWarp) {
    if (n >= 1) {
      const int32_t x = tokens[(int64_t)b * M + n];
      bad_tok |= (x < 0 || x >= V);
    }
    const RowNorm t = ld_norm(nb + n);
    bad_row |= !(t.m > -INFINITY && t.m < INFINITY && t.S > 0.0 && t.S < INFINITY);
    if (n < M - 1) {
      const RowNorm q = ld_norm(nb + M + n);
      bad_row |= !(q.m > -INFINITY && q.m < INFINITY && q.S > 0.0 && q.S < INFINITY);
    }
  }
  bad_arg = __any_sync(0xffffffffu, bad_arg);
  bad_tok = __any_sync(0xffffffffu, bad_tok);
  bad_row = __any_sync(0xffffffffu, bad_row);
  if (bad_arg || bad_tok || bad_row) {
    for (int i = lane; i < M; i += kWarp) {
      ot[i] = -1;
      pt[i] = -1;
    }
    if (pr != nullptr)
      for (int i = lane; i < 4 * M; i += kWarp) pr[i] = -1.f;
    if (lane == 0) {
      accepted_len[b] = -1;
      raise_status(w.status, bad_arg ? SPEC_ERR_INVALID_ARG
                             : bad_tok ? SPEC_ERR_DEVICE_BOUNDS
                                       : SPEC_ERR_NONFINITE);
    }
    fused_finish(w.ctl);
    return;
  }

  // the accept tests: lane n - 1 (mod 32) tests draft n against row n - 1
  const uint64_t bglob = b_base + (uint64_t)b;
  const double cs64 = (double)cs;
  int fr = M;  // first rejected draft, M if none
  for (int n0 = 1; n0 < M && fr == M; n0 += kWarp) {
    const int n = n0 + lane;
    bool rej = false;
    float pp = -1.f, qq = -1.f;
    if (n < M) {
      const int p = n - 1;
      const int32_t x = tokens[(int64_t)b * M + n];
      const int64_t o = ((int64_t)b * M + p) * V + x;
      const float zt = to_f32(target[o]), zd = to_f32(draft[o]);
      const RowNorm t = ld_norm(nb + p), q = ld_norm(nb + M + p);
      if (greedy) {
        rej = x != t.amax;
        pp = rej ? 0.f : 1.f;
        qq = x == q.amax ? 1.f : 0.f;
      } else {
        const Philox4 r = philox4x64_10((uint64_t)n + 1, bglob, offset, 0, seed, 0);
        const float uacc = (float)u24(r.w[0]);
        const double et = ((double)zt - (double)t.m) * cs64;  // log2 unnormalised p(x)
        const double ed = ((double)zd - (double)q.m) * cs64;  // log2 unnormalised q(x)
        const float st_f = (float)t.S, sd_f = (float)q.S;
        bool acc;
        if (ed == -INFINITY) {
          acc = et != -INFINITY;
        } else if (et == -INFINITY) {
          acc = false;
        } else {
          const double e = et - ed;
          const double ei = rint(e);
          const float ratio =
              ldexpf(fast_exp2((float)(e - ei)), (int)fmax(fmin(ei, 300.0), -300.0)) * (sd_f / st_f);
          acc = uacc < ratio;
        }
        rej = !acc;
        pp = exp2f((float)et) / st_f;
        qq = exp2f((float)ed) / sd_f;
      }
    }
    const unsigned rb = __ballot_sync(0xffffffffu, rej);
    const int first = rb ? n0 + __ffs(rb) - 1 : M;
    // probes of the tested drafts: up to and including the first rejected
    if (pr != nullptr && n < M) {
      const bool tested = n <= first;
      pr[n * 4 + 0] = tested ? pp : -1.f;
      pr[n * 4 + 1] = tested ? qq : -1.f;
      pr[n * 4 + 2] = -1.f;
      pr[n * 4 + 3] = -1.f;
    }
    if (first < M) fr = first;
  }
  if (pr != nullptr) {
    for (int n = fr + 1 + lane; n < M; n += kWarp) {  // past the first rejection: untested
      pr[n * 4 + 0] = -1.f;
      pr[n * 4 + 1] = -1.f;
      pr[n * 4 + 2] = -1.f;
      pr[n * 4 + 3] = -1.f;
    }
    if (lane == 0)
      for (int i = 0; i < 4; ++i) pr[i] = -1.f;  // the root is never tested
  }
  const int a = fr < M ? fr - 1 : M - 1;  // accepted drafts = the node that draws
  for (int n = lane; n < M; n += kWarp) {
    pt[n] = n <= a ? n : -1;
    if (n < a) ot[n] = tokens[(int64_t)b * M + n + 1];
    else if (n > a) ot[n] = -1;
  }
  if (lane == 0) accepted_len[b] = a;

  if (greedy) {
    // the token at node a is its target row's first largest logit
    if (lane == 0) {
      ot[a] = ld_norm(nb + a).amax;
      if (pr != nullptr) {
        pr[a * 4 + 2] = 1.f;
        pr[a * 4 + 3] = 1.f;
      }
    }
    fused_finish(w.ctl);
    return;
  }
  const Philox4 r = philox4x64_10((uint64_t)a + 1, bglob, offset, 0, seed, 0);
  const double u = (double)u24(r.w[1]);
  const RowNorm ta = ld_norm(nb + a);
  DecideCtx c;
  ctx_no_filter(c);
  c.mT = ta.m;
  c.invST = (float)(1.0 / ta.S);
  c.cs = cs;
  if (fr < M) {
    // the residual max(0, p_a - q_a): post its chunks
    const RowNorm da = ld_norm(nb + M + a);
    c.mD = da.m;
    c.invSD = (float)(1.0 / da.S);
    c.nrej = 1;
    if (lane == 0) {
      const uint32_t e = atomicAdd(w.ctl + kCEntries, 1u);
      ResEntry* r = w.entries + e;
      r->b = b;
      r->node = a;
      r->a = a;
      r->mT = c.mT;
      r->mD = c.mD;
      r->invST = c.invST;
      r->invSD = c.invSD;
      r->cs = c.cs;
      r->u = u;
      __threadfence();
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&r->ready), "r"(1u) : "memory");
      atomicAdd(w.ctl + kCPub, (uint32_t)((n_chunks + kFUnit - 1) / kFUnit));
    }
    return;
  }
  // every draft accepted: the bonus token from p of the last node
  c.mD = 0.f;
  c.invSD = 0.f;
  c.nrej = 0;
  const T* trow = target + ((int64_t)b * M + a) * V;
  const RowStat* tst = w.stats + (((int64_t)b * 2 + 0) * M + a) * n_chunks;
  float wt;
  double z;
  const int tk = warp_draw_from_p<T>(trow, tst, n_chunks, chunk, V, c, u, &wt, &z);
  if (lane == 0) {
    ot[a] = tk;
    if (pr != nullptr) {
      pr[a * 4 + 2] = 1.0f;
      pr[a * 4 + 3] = (float)((double)wt / z);
    }
  }
  fused_finish(w.ctl);
}

// One residual unit (entry e, chunk group g: statistics chunks
// [kFUnit g, kFUnit g + kFUnit)), by one warp: each chunk's residual mass;
// the unit that completes its request draws the token.
template <typename T>
__device__ __noinline__ bool fused_residual_unit(const T* __restrict__ target,
                                                 const T* __restrict__ draft,
                                                 int32_t* __restrict__ out_tokens,
                                                 float* __restrict__ probe, const spec_dims& d,
                                                 int n_chunks, int chunk, const FusedWs& w,
                                                 uint32_t e, int g, volatile int* abort,
                                                 uint64_t wait) {
  const int lane = threadIdx.x % kWarp;
  const int M = d.M, V = d.V;
  ResEntry* ent = w.entries + e;
  // the entry is allocated; its writer publishes it right away (bounded)
  if (lane == 0) {
    long long t0 = 0;
    for (uint32_t it = 0; ld_acquire_u32(&ent->ready) == 0u; ++it) {
      if ((it & 15u) == 15u) {
        if (*abort || ld_relaxed_u32(w.ctl + kCFail) != 0u) {
          *abort = 1;
          break;
        }
        const long long now = clock64();
        if (t0 == 0) {
          t0 = now;
        } else if ((uint64_t)(now - t0) > wait) {
          *abort = 1;
          break;
        }
      }
      __nanosleep(64);
    }
  }
  if (__shfl_sync(0xffffffffu, (int)*abort, 0)) return false;
  const uint4 r0 = __ldcg(reinterpret_cast<const uint4*>(ent));
  const uint4 r1 = __ldcg(reinterpret_cast<const uint4*>(ent) + 1);
  const uint4 r2 = __ldcg(reinterpret_cast<const uint4*>(ent) + 2);
  const int b = (int)r0.x, node = (int)r0.y, a_acc = (int)r0.z;
  DecideCtx ctx;
  ctx_no_filter(ctx);
  ctx.mT = __uint_as_float(r1.x);
  ctx.mD = __uint_as_float(r1.y);
  ctx.invST = __uint_as_float(r1.z);
  ctx.invSD = __uint_as_float(r1.w);
  ctx.cs = __uint_as_float(r2.x);
  ctx.nrej = 1;
  const double u = __hiloint2double((int)r2.w, (int)r2.z);
  const T* trow = target + ((int64_t)b * M + node) * V;
  const T* drow = draft + ((int64_t)b * M + node) * V;
  double* zs = w.zsum + (int64_t)b * n_chunks;
  const int c1 = min(n_chunks, (g + 1) * kFUnit);
  for (int c = g * kFUnit; c < c1; ++c) {
    uint4 raw_t[kStatVecs], raw_d[kStatVecs];
    const float ls = lane_weights<T, false>(trow, drow, (int64_t)c * chunk, V, ctx, 1, raw_t, raw_d);
    const dfloat tot = df_warp_sum(df_make(ls));
    if (lane == 0) zs[c] = df_to_d(tot);
  }
  const uint32_t n_units = (uint32_t)((n_chunks + kFUnit - 1) / kFUnit);
  uint32_t done = 0;
  if (lane == 0) {
    __threadfence();
    done = atomicAdd(w.res_cnt + b, 1u) + 1u;
  }
  done = __shfl_sync(0xffffffffu, done, 0);
  if (done != n_units) return true;
  // the last unit of request b: the draw
  __threadfence();
  double Z = 0.0;
  for (int k = lane; k < n_chunks; k += kWarp) Z += __ldcg(zs + k);
  Z = warp_sum(Z);
  float wt;
  int tk;
  double zrep;
  if (Z > 0.0) {
    double pre;
    const int sel = warp_select_chunk(zs, n_chunks, u * Z, &pre);
    const double trel = u * Z - pre;
    const float th = (float)trel;
    tk = warp_chunk_draw<T, false>(trow, drow, (int64_t)sel * chunk, V, ctx, 1,
                            dfloat{th, (float)(trel - (double)th)}, &wt);
    zrep = Z;
  } else {
    // a residual of zero mass: the draw from p of the node
    DecideCtx cp = ctx;
    cp.nrej = 0;
    const RowStat* tst = w.stats + (((int64_t)b * 2 + 0) * M + node) * n_chunks;
    double z;
    tk = warp_draw_from_p<T>(trow, tst, n_chunks, chunk, V, cp, u, &wt, &z);
    zrep = z;
    Z = 1.0;
  }
  if (lane == 0) {
    out_tokens[(int64_t)b * M + a_acc] = tk;
    if (probe != nullptr) {
      probe[((int64_t)b * M + node) * 4 + 2] = (float)Z;
      probe[((int64_t)b * M + node) * 4 + 3] = (float)((double)wt / zrep);
    }
    w.res_cnt[b] = 0u;  // ready for the next call
  }
  fused_finish(w.ctl);
  return true;
}

template <typename T>
__global__ void __launch_bounds__(kFWarps * kWarp, 1) rs_fused_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const float* __restrict__ temperature, uint64_t seed, uint64_t offset, uint64_t b_base,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ path,
    int32_t* __restrict__ accepted_len, float* __restrict__ probe, spec_dims d, int n_chunks,
    int chunk, FusedWs w) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kChunk = kWarp * kStatVecs * EPV;
  __shared__ uint64_t full[kFWarps][kFRing];
  __shared__ long long s_task[kFWarps][kFRing];
  __shared__ int s_abort, s_last;
  // the control words [kCPub..kCFail] as last read by a warp of this CTA, and
  // when: idle warps read them here instead of from L2
  __shared__ uint32_t s_cw[4];
  __shared__ long long s_cw_time;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const int B = d.B, M = d.M, V = d.V;
  const uint64_t wait = wait_limit_cycles(d);
  if (tid == 0) {
    for (int i = 0; i < kFWarps; ++i)
      for (int j = 0; j < kFRing; ++j) ptx::mbar_init(ptx::smem_u32(&full[i][j]), 1);
    s_abort = 0;
    s_cw[0] = s_cw[1] = s_cw[2] = s_cw[3] = 0u;
    s_cw_time = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // the logits may come from the previous kernel
  volatile int* abort = &s_abort;
  volatile uint32_t* cws = s_cw;
  volatile long long* cw_time = &s_cw_time;
  uint32_t* ctl = w.ctl;
  const int rows = 2 * M - 1;  // target rows 0..M-1, then draft rows 0..M-2
  const int64_t per_req = (int64_t)rows * n_chunks;
  const int64_t ntask = per_req * B;
  const int64_t nbatch = (ntask + kFBatch - 1) / kFBatch;
  const uint32_t n_units = (uint32_t)((n_chunks + kFUnit - 1) / kFUnit);
  uint8_t* myring = ring + (size_t)warp * kFRing * kBulkSlot;
  uint64_t* mybars = full[warp];
  long long* mytask = s_task[warp];
  // warps 0..3 of each CTA take residual units between their batches
  const bool poll = warp < 4;

  // the control words, from L2 (lane 0), kept in shared memory for the CTA
  auto load_cw = [&](uint4& cw) {
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(cw.x), "=r"(cw.y), "=r"(cw.z), "=r"(cw.w)
                 : "l"(ctl + kCPub)
                 : "memory");
  };

  // the stream: tasks [it, it_end) of the current batch are still to be
  // issued; lane 0's `next` is the batch claimed after it (claimed one batch
  // early, so that the atomic's latency hides behind the copies)
  int64_t it = 0, it_end = 0;
  uint32_t next = 0;
  if (lane == 0) next = atomicAdd(ctl + kCBatch, 1u);
  bool stream_done = false;
  int64_t issued = 0, consumed = 0;
  auto issue_one = [&]() -> bool {  // whole warp; false once the stream has no task left
    if (it == it_end) {
      const uint32_t nb = __shfl_sync(0xffffffffu, next, 0);
      if ((int64_t)nb >= nbatch) return false;
      it = (int64_t)nb * kFBatch;
      it_end = it + kFBatch < ntask ? it + kFBatch : ntask;
      if (lane == 0) next = atomicAdd(ctl + kCBatch, 1u);
    }
    const int64_t t = it++;
    const int slot = (int)(issued % kFRing);
    if (lane == 0) {
      const int b = (int)(t / per_req);
      const int rem = (int)(t - (int64_t)b * per_req);
      const int row = rem / n_chunks, c = rem - row * n_chunks;
      const T* src = row < M ? target + ((int64_t)b * M + row) * V
                             : draft + ((int64_t)b * M + (row - M)) * V;
      const int64_t e0 = (int64_t)c * kChunk;
      const int64_t left = (int64_t)V - e0;
      const uint32_t bytes = (uint32_t)((left < kChunk ? left : kChunk) * sizeof(T));
      mytask[slot] = t;
      const uint32_t bar = ptx::smem_u32(&mybars[slot]);
      ptx::mbar_arrive_expect_tx(bar, bytes);
      ptx::bulk_g2s(ptx::smem_u32(myring + (size_t)slot * kBulkSlot), src + e0, bytes, bar);
    }
    ++issued;
    return true;
  };

  // Finished chunks of one row not yet counted (acc_*), and the count added
  // last whose returned value is still to be looked at (pend_*: lane 0's
  // atomic result, read one batch later).
  int acc_key = -1, acc_b = 0;
  uint32_t acc_n = 0;
  float acc_cs = 1.f;
  int pend_key = -1, pend_b = 0;
  uint32_t pend_n = 0, pend_old = 0;
  float pend_cs = 1.f;
  // Looks at the pending count: the warp whose chunks complete a row forms
  // its normaliser; the row that completes a request has it decided.
  auto resolve = [&]() {  // whole warp
    if (pend_n == 0) return;
    const uint32_t old = __shfl_sync(0xffffffffu, pend_old, 0);
    const uint32_t n = pend_n;
    pend_n = 0;
    if (old + n != (uint32_t)n_chunks) return;
    __threadfence();
    const int b = pend_b, row = pend_key - b * 2 * M;
    const int which = row < M ? 0 : 1, node = row < M ? row : row - M;
    fused_row_norm(w.stats + (((int64_t)b * 2 + which) * M + node) * n_chunks, n_chunks, chunk,
                   pend_cs, w.norms + pend_key);
    uint32_t r = 0;
    if (lane == 0) {
      w.row_cnt[pend_key] = 0u;  // ready for the next call
      __threadfence();
      r = atomicAdd(w.req_rows + b, 1u) + 1u;
    }
    r = __shfl_sync(0xffffffffu, r, 0);
    if (r != (uint32_t)rows) return;
    __threadfence();
    if (lane == 0) w.req_rows[b] = 0u;
    fused_decide<T>(target, draft, tokens, temperature, seed, offset, b_base, out_tokens, path,
                    accepted_len, probe, d, n_chunks, chunk, w, b);
  };
  // Adds the accumulated count to its row (after this warp's statistics are
  // visible); the previous pending count is looked at first.
  auto flush = [&]() {  // whole warp
    if (acc_n == 0) return;
    resolve();
    if (lane == 0) {
      __threadfence();
      pend_old = atomicAdd(w.row_cnt + acc_key, acc_n);
    }
    pend_key = acc_key;
    pend_b = acc_b;
    pend_n = acc_n;
    pend_cs = acc_cs;
    acc_n = 0;
  };

  int64_t reserved = -1;  // a residual unit this warp claimed and has not done
  // Claims a unit when some are published and unclaimed, and does the one
  // held once it is published.  Returns false if a wait gave up.
  auto take_units = [&](uint32_t pub, uint32_t clm, bool* progressed) -> bool {
    if (reserved < 0 && pub > clm) {
      uint32_t u = 0;
      if (lane == 0) u = atomicAdd(ctl + kCClaim, 1u);
      reserved = (int64_t)__shfl_sync(0xffffffffu, u, 0);
    }
    if (reserved >= 0 && (uint64_t)reserved < (uint64_t)pub) {
      const uint32_t e = (uint32_t)(reserved / n_units);
      const int g = (int)(reserved - (int64_t)e * n_units);
      reserved = -1;
      *progressed = true;
      return fused_residual_unit<T>(target, draft, out_tokens, probe, d, n_chunks, chunk, w, e, g,
                                    abort, wait);
    }
    return true;
  };

  // ---- the stream ---------------------------------------------------------
  int cur_b = -1;
  float cs = 1.f;
  bool greedy = false;
  bool ok = true;
  while (ok) {
    if (*abort) {
      ok = false;
      break;
    }
    while (!stream_done && issued - consumed < kFRing)
      if (!issue_one()) stream_done = true;
    if (consumed == issued) break;  // nothing left to stream for this warp
    // the control words, loaded now and looked at after the batch
    uint4 cw = make_uint4(0, 0, 0, 0);
    if (lane == 0 && poll) load_cw(cw);
    for (int k = 0; k < kFBatch && consumed < issued; ++k) {
      const int slot = (int)(consumed % kFRing);
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&mybars[slot]),
                                                   (uint32_t)((consumed / kFRing) & 1), abort,
                                                   wait))) {
        ok = false;
        break;
      }
      const int64_t t = mytask[slot];
      const int b = (int)(t / per_req);
      const int rem = (int)(t - (int64_t)b * per_req);
      const int row = rem / n_chunks, c = rem - row * n_chunks;
      if (b != cur_b) {
        cur_b = b;
        const float temp = temperature[b];
        cs = stat_scale(temp);
        greedy = temp == 0.f;
      }
      const int e0 = c * kChunk;
      const int nvalid = V - e0;
      const uint4* sv = reinterpret_cast<const uint4*>(myring + (size_t)slot * kBulkSlot);
      uint4 raw[kStatVecs];
#pragma unroll
      for (int v = 0; v < kStatVecs; ++v) raw[v] = sv[v * kWarp + lane];
      float sd;
      const float m = chunk_stat<T>(raw, nvalid, cs, &sd);
      const int am = greedy ? chunk_argmax<T>(raw, nvalid, m) : 0;
      const int which = row < M ? 0 : 1, node = row < M ? row : row - M;
      if (lane == 0) {
        RowStat r;
        r.m = m;
        r.pad = pack_index(am);
        r.s = (double)sd;
        w.stats[(((int64_t)b * 2 + which) * M + node) * n_chunks + c] = r;
      }
      ++consumed;
      __syncwarp();
      // the slot's reads are done before the async proxy refills it
      ptx::fence_proxy_async_smem();
      if (!stream_done && !issue_one()) stream_done = true;
      const int key = b * 2 * M + row;
      if (key != acc_key) {
        flush();
        acc_key = key;
        acc_b = b;
        acc_cs = cs;
      }
      ++acc_n;
    }
    if (!ok) break;
    flush();
    if (poll) {
      const uint32_t pub = __shfl_sync(0xffffffffu, cw.x, 0);
      const uint32_t clm = __shfl_sync(0xffffffffu, cw.y, 0);
      const uint32_t fail = __shfl_sync(0xffffffffu, cw.w, 0);
      if (fail != 0u) {
        *abort = 1;
        ok = false;
        break;
      }
      bool prog = false;
      if (!take_units(pub, clm, &prog)) ok = false;
    }
  }
  // the stream is over for this warp: its last count is looked at
  if (ok && !*abort) {
    flush();
    resolve();
  }

  // ---- after the stream: residual units until every request is finished --
  long long idle0 = 0;
  int backoff = 32;
  while (ok && !*abort) {
    uint4 cw;
    const long long now = clock64();
    if (warp == 0 || now - *cw_time > 2000) {
      // this CTA's copy is old: read the words from L2
      if (lane == 0) {
        load_cw(cw);
        cws[0] = cw.x;
        cws[1] = cw.y;
        cws[2] = cw.z;
        cws[3] = cw.w;
        *cw_time = now;
      }
    } else if (lane == 0) {
      cw = make_uint4(cws[0], cws[1], cws[2], cws[3]);
    }
    const uint32_t pub = __shfl_sync(0xffffffffu, cw.x, 0);
    const uint32_t clm = __shfl_sync(0xffffffffu, cw.y, 0);
    const uint32_t fin = __shfl_sync(0xffffffffu, cw.z, 0);
    const uint32_t fail = __shfl_sync(0xffffffffu, cw.w, 0);
    if (fail != 0u) {
      *abort = 1;
      break;
    }
    if (fin >= (uint32_t)B) break;
    bool prog = false;
    if (!take_units(pub, clm, &prog)) break;
    if (prog) {
      idle0 = 0;
      backoff = 32;
      continue;
    }
    const long long t = clock64();
    if (idle0 == 0) {
      idle0 = t;
    } else if ((uint64_t)(t - idle0) > wait) {
      *abort = 1;
      break;
    }
    __nanosleep(backoff);
    backoff = backoff < 512 ? 2 * backoff : 512;
  }
  // a wait that gave up fails the call for every CTA at once
  if (lane == 0 && *abort) atomicExch(ctl + kCFail, 1u);
  // copies issued but not consumed (only after a wait gave up) land before
  // the CTA exits; these waits ignore the abort flag and keep their own limit
  if (lane == 0)
    for (int64_t u = consumed; u < issued; ++u)
      ptx::mbar_drain(ptx::smem_u32(&mybars[u % kFRing]), (uint32_t)((u / kFRing) & 1),
                      kDefaultWaitCycles);
  __syncthreads();
  if (tid == 0 && *abort) raise_status(w.status, SPEC_ERR_TIMEOUT);
  // the last CTA out: a failed call fails every request; the counters go
  // back to zero for the next call
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(ctl + kCCtas, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    const uint32_t ne = ld_relaxed_u32(ctl + kCEntries);
    const bool failed = ld_relaxed_u32(ctl + kCFail) != 0u;
    for (uint32_t e = tid; e < ne && e < (uint32_t)B; e += blockDim.x) w.entries[e].ready = 0u;
    if (failed)
      for (int b = tid; b < B; b += blockDim.x) accepted_len[b] = -1;
    __syncthreads();
    if (tid == 0) {
      ctl[kCBatch] = 0u;
      ctl[kCEntries] = 0u;
      ctl[kCPub] = 0u;
      ctl[kCClaim] = 0u;
      ctl[kCFin] = 0u;
      ctl[kCFail] = 0u;
      __threadfence();
      ctl[kCCtas] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
template <typename T, bool kAligned>
static cudaError_t launch_rs_t(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  const spec_dims& d = a.d;
  char* ws = static_cast<char*>(a.ws);
  RowStat* stats = reinterpret_cast<RowStat*>(ws + lay.rs_off);
  DrawState* draws = reinterpret_cast<DrawState*>(ws + lay.rs_draw_off);
  double* zsum = reinterpret_cast<double*>(ws + lay.rs_zsum_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + lay.status_off);
  const T* tgt = static_cast<const T*>(a.target);
  const T* dft = static_cast<const T*>(a.draft);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ntask = (int64_t)lay.rs_chunks * 2 * d.M * d.B;
  const int64_t want = (ntask + kRsThreads / kWarp - 1) / (kRsThreads / kWarp);
  if (a.stats_ready) {
    // the LM head wrote the statistics
  } else if (kAligned) {
    const int64_t wantb = (ntask + kBulkWarps - 1) / kBulkWarps;
    const unsigned gb = (unsigned)(wantb < sms ? wantb : sms);
    // A chain's last tasks as a pool (the two counters after the tail's),
    // when the warps have many tasks each (24 or more): then the stream's
    // end is uneven across SMs.  With few, the equal ceil-sized ranges
    // leave the last SMs idle early, and the kernel after this one starts
    // its CTAs there (measured: the pool is 6% faster at 35 tasks per warp,
    // 3% slower at 14).
    const int64_t per_warp = ntask / ((int64_t)gb * kBulkWarps);
    uint32_t* pool = a.parent == nullptr && per_warp >= 24
                         ? reinterpret_cast<uint32_t*>(ws + lay.rs_tail_off) + 2 * (size_t)d.B
                         : nullptr;
    cudaError_t e;
    if (pool != nullptr) {
      e = cudaFuncSetAttribute(rs_rowstats_pool_kernel<T>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPoolSmem);
      if (e != cudaSuccess) return e;
      PdlLaunch L(dim3(gb), dim3(kBulkWarps * kWarp), kPoolSmem, st);
      e = cudaLaunchKernelEx(&L.cfg, rs_rowstats_pool_kernel<T>, tgt, dft, a.parent,
                             a.temperature, d, lay.rs_chunks, stats, status, pool);
    } else {
      e = cudaFuncSetAttribute(rs_rowstats_bulk_kernel<T>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem);
      if (e != cudaSuccess) return e;
      PdlLaunch L(dim3(gb), dim3(kBulkWarps * kWarp), kBulkSmem, st);
      e = cudaLaunchKernelEx(&L.cfg, rs_rowstats_bulk_kernel<T>, tgt, dft, a.parent,
                             a.temperature, d, lay.rs_chunks, stats, status);
    }
    if (e != cudaSuccess) return e;
  } else {
    const unsigned g1 = (unsigned)(want < 2 * sms ? want : 2 * sms);
    PdlLaunch L(dim3(g1), dim3(kRsThreads), 0, st);
    const cudaError_t e = cudaLaunchKernelEx(&L.cfg, rs_rowstats_kernel<T, false>, tgt, dft,
                                             a.parent, a.temperature, d, lay.rs_chunks, stats);
    if (e != cudaSuccess) return e;
  }
  // a chain of aligned, unfiltered rows: the whole tail in one launch
  if (kAligned && a.parent == nullptr && a.top_k == nullptr && a.top_p == nullptr) {
    // about eight chunks of the residual per slice (one per warp), and no
    // more CTAs than fit on the GPU at once (two per SM)
    const int want_s = (lay.rs_chunks + 7) / 8;
    const int cap_s = (2 * sms) / d.B > 1 ? (2 * sms) / d.B : 1;
    int S = want_s < cap_s ? want_s : cap_s;
    if (S > 16) S = 16;
    if (S < 1) S = 1;
    PdlLaunch L(dim3((unsigned)((int64_t)d.B * S)), dim3(kTailThreads), 0, st);
    const cudaError_t e = cudaLaunchKernelEx(
        &L.cfg, rs_chain_tail_kernel<T>, tgt, dft, a.tokens, a.temperature, a.seed, a.offset,
        a.b_base, a.out_tokens, a.path, a.accepted_len, a.probe, d, lay.rs_chunks, lay.rs_chunk,
        (const RowStat*)stats, zsum, reinterpret_cast<uint32_t*>(ws + lay.rs_tail_off), status, S,
        a.stats_ready ? 0 : 1);
    if (e != cudaSuccess) return e;
    *launches += a.stats_ready ? 1 : 2;
    return cudaGetLastError();
  }
  // a tree of aligned, unfiltered rows: the walk by clusters, beside the
  // statistics pass (after the LM heads it waits for them first)
  if (rs_tree_walk_supported(d, kAligned, a.parent != nullptr,
                             a.top_k != nullptr || a.top_p != nullptr)) {
    const cudaError_t e = rs_tree_walk_launch(a, lay, !a.stats_ready, st);
    if (e != cudaSuccess) return e;
    *launches += a.stats_ready ? 1 : 2;
    return cudaGetLastError();
  }
  // passes 2 and 3 start while their predecessor drains (programmatic
  // dependent launch); each waits for its predecessor's results in-kernel
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)d.B);
  // filtered laws (top-k / top-p): each row's kept prefix, after the
  // statistics and before the decisions
  const bool filters = a.top_k != nullptr || a.top_p != nullptr;
  FilterInfo* finfo = filters ? reinterpret_cast<FilterInfo*>(ws + lay.rs_filt_off) : nullptr;
  cudaError_t e;
  if (filters) {
    cfg.blockDim = dim3(kFiltThreads);
    cfg.gridDim = dim3((unsigned)(2 * d.M), (unsigned)d.B);
    e = cudaLaunchKernelEx(&cfg, rs_filter_kernel<T, kAligned>, tgt, dft, a.parent, a.temperature,
                           a.top_k, a.top_p, d, lay.rs_chunks, (const RowStat*)stats, finfo);
    if (e != cudaSuccess) return e;
    ++*launches;
    cfg.blockDim = dim3(kDecThreads);
    cfg.gridDim = dim3((unsigned)d.B);
  }
  e = cudaLaunchKernelEx(&cfg, rs_decide_kernel<T, kAligned>, tgt, dft, a.tokens, a.parent,
                         a.temperature, a.seed, a.offset, a.b_base, a.out_tokens, a.path,
                         a.accepted_len, a.probe, d, lay.rs_chunks, lay.rs_chunk,
                         (const RowStat*)stats, draws, status, a.top_k, a.top_p,
                         (const FilterInfo*)finfo);
  if (e != cudaSuccess) return e;
  cfg.blockDim = dim3(kResThreads);
  cfg.gridDim = dim3((unsigned)((int64_t)rs_res_spans(lay.rs_chunks) * d.B));
  e = cudaLaunchKernelEx(&cfg, rs_residual_sums_kernel<T, kAligned>, tgt, dft, d, lay.rs_chunks,
                         lay.rs_chunk, (const DrawState*)draws, zsum);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)d.B);
  e = cudaLaunchKernelEx(&cfg, rs_residual_draw_kernel<T, kAligned>, tgt, dft, d, lay.rs_chunks,
                         lay.rs_chunk, (const RowStat*)stats, (const DrawState*)draws,
                         (const double*)zsum, a.out_tokens, a.probe);
  if (e != cudaSuccess) return e;
  *launches += a.stats_ready ? 3 : 4;
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_fused_t(const RsArgs& a, const WsLayout& lay, cudaStream_t st,
                                  int* launches) {
  const spec_dims& d = a.d;
  char* ws = static_cast<char*>(a.ws);
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(rs_fused_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kFSmem);
  if (e != cudaSuccess) return e;
  FusedWs w;
  w.stats = reinterpret_cast<RowStat*>(ws + lay.rs_off);
  w.norms = reinterpret_cast<RowNorm*>(ws + lay.rsf_norm_off);
  w.row_cnt = reinterpret_cast<uint32_t*>(ws + lay.rsf_rowcnt_off);
  w.req_rows = reinterpret_cast<uint32_t*>(ws + lay.rsf_req_off);
  w.entries = reinterpret_cast<ResEntry*>(ws + lay.rsf_list_off);
  w.res_cnt = reinterpret_cast<uint32_t*>(ws + lay.rsf_rescnt_off);
  w.zsum = reinterpret_cast<double*>(ws + lay.rs_zsum_off);
  w.ctl = reinterpret_cast<uint32_t*>(ws + lay.rsf_ctl_off);
  w.status = reinterpret_cast<uint32_t*>(ws + lay.status_off);
  PdlLaunch L(dim3(sms), dim3(kFWarps * kWarp), kFSmem, st);
  e = cudaLaunchKernelEx(&L.cfg, rs_fused_kernel<T>, static_cast<const T*>(a.target),
                         static_cast<const T*>(a.draft), a.tokens, a.temperature, a.seed, a.offset,
                         a.b_base, a.out_tokens, a.path, a.accepted_len, a.probe, d, lay.rs_chunks,
                         lay.rs_chunk, w);
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaGetLastError();
}

size_t rsf_layout(const spec_dims& d, size_t off, WsLayout* L) {
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = (off + bytes + 255) / 256 * 256;
    return o;
  };
  const size_t rows = (size_t)d.B * 2 * d.M;
  L->rsf_ctl_off = take(sizeof(uint32_t) * kFCtl);
  L->rsf_norm_off = take(sizeof(RowNorm) * rows);
  L->rsf_rowcnt_off = take(sizeof(uint32_t) * rows);
  L->rsf_req_off = take(sizeof(uint32_t) * (size_t)d.B);
  L->rsf_list_off = take(sizeof(ResEntry) * (size_t)d.B);
  L->rsf_rescnt_off = take(sizeof(uint32_t) * (size_t)d.B);
  return off;
}

bool rso_supported(const spec_dims& d, bool aligned, bool chain) {
  return aligned && chain && d.M <= kMaxM;
}

cudaError_t rs_launch(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  const int esz = a.d.logits_dtype == SPEC_BF16 ? 2 : 4;
  const bool aligned = ((size_t)a.d.V * esz) % 16 == 0 &&
                       (reinterpret_cast<uintptr_t>(a.target) % 16) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.draft) % 16) == 0;
  // the one-kernel path takes neither trees nor filters
  const bool fused_ok = rso_supported(a.d, aligned, a.parent == nullptr) &&
                        a.top_k == nullptr && a.top_p == nullptr;
  if (a.d.reject_impl == SPEC_REJECT_FUSED) {
    if (!fused_ok) return cudaErrorNotSupported;
    return a.d.logits_dtype == SPEC_BF16 ? launch_fused_t<__nv_bfloat16>(a, lay, st, launches)
                                         : launch_fused_t<float>(a, lay, st, launches);
  }
  if (a.d.logits_dtype == SPEC_BF16)
    return aligned ? launch_rs_t<__nv_bfloat16, true>(a, lay, st, launches)
                   : launch_rs_t<__nv_bfloat16, false>(a, lay, st, launches);
  return aligned ? launch_rs_t<float, true>(a, lay, st, launches)
                 : launch_rs_t<float, false>(a, lay, st, launches);
}

}  // namespace specv
