// The verify walk of a tree by a cluster of CTAs per request, beside the
// statistics pass.
//
// Method (page 3, formal definition and tree-attention section; page 1
// §4.1): at node n the children are tried in ascending order; child c with
// drafted token x is accepted iff u * Q(x) < P(x), where P starts as the
// target law p_n and every rejected child turns it into
// normalize(max(0, P - q_n)); an accepted child becomes the node, and a
// node where no child is accepted (or that has none) draws one token from P
// by the inverse CDF in vocabulary order.  Temperature 0 is the point-mass
// reading (exact match with each row's first argmax).
//
// The decisions need only the rows the walk visits -- a few of the tree's
// nodes -- so a cluster of kTwCtas CTAs walks each request: CTA r owns slice
// r of every row (1/kTwCtas of the vocabulary, whole 16-byte vectors).  Per
// visited node, one exchange through distributed shared memory gives every
// CTA the node's normalisers (the slices' maxima and sums, combined the same
// way in every CTA), each rejected child one more exchange for the
// residual's mass,
// and the draw's slice is searched by the CTA that owns it.  Every CTA makes
// the same decisions from the same exchanged values.  An exchange is eight
// remote stores and eight remote mbarrier arrivals per CTA, and a bounded
// wait on the CTA's own mbarrier: no wait can hang.
//
// The statistics pass over every row still decides which requests fail (a
// row with NaN, +inf or only -inf, visited or not), but the walk does not
// wait for it: the statistics kernel lets this kernel launch once all the
// work before it on the stream has completed, so the walk reads its inputs
// at once and runs beside the statistics stream; only the final verdict
// waits for the statistics.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "philox.cuh"
#include "reject_sample.cuh"
#include "rs_device.cuh"
#include "tc_ptx.cuh"

namespace specv {

constexpr int kTwCtas = 8;  // CTAs per request (one cluster)
constexpr int kTwThreads = 256;
constexpr int kTwWarps = kTwThreads / kWarp;
constexpr int kTwBatch = 4;  // 16-byte vectors of a row loaded together per thread

namespace tw {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_remote_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Running (maximum, sum of exp2((z - max) cs), first index of the maximum)
// of a stream of logits in increasing index order.
struct Run {
  float m, s;
  int a;
};
__device__ __forceinline__ void run_add(Run& r, float z, int e, float cs) {
  if (z > r.m) {
    r.s = (r.m == -INFINITY ? 0.f : r.s * fast_exp2((r.m - z) * cs)) + 1.f;
    r.m = z;
    r.a = e;
  } else if (z != -INFINITY) {
    r.s += fast_exp2((z - r.m) * cs);
  }
}
// Merge of two runs over interleaved index sets.
__device__ __forceinline__ Run run_merge(Run x, Run y, float cs) {
  Run o;
  o.m = fmaxf(x.m, y.m);
  o.s = (x.m == -INFINITY ? 0.f : x.s * fast_exp2((x.m - o.m) * cs)) +
        (y.m == -INFINITY ? 0.f : y.s * fast_exp2((y.m - o.m) * cs));
  o.a = x.m == y.m ? min(x.a, y.a) : (x.m > y.m ? x.a : y.a);  // first index on ties
  if (o.m != o.m) o.a = 0;  // NaN: the row fails later
  return o;
}
__device__ __forceinline__ Run run_warp(Run r, float cs) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Run y;
    y.m = __shfl_xor_sync(0xffffffffu, r.m, o);
    y.s = __shfl_xor_sync(0xffffffffu, r.s, o);
    y.a = __shfl_xor_sync(0xffffffffu, r.a, o);
    r = run_merge(r, y, cs);
  }
  return r;
}

// 2^e for e in fp64 (formed exactly from fp32 operands): the integer part
// by scaling, the fraction by the fp32 exp2 (about 1e-7 relative).
__device__ __forceinline__ double exp2_split(double e) {
  if (e == -INFINITY) return 0.0;
  const double ei = rint(e);
  const int k = (int)fmax(fmin(ei, 1000.0), -1100.0);
  return ldexp((double)exp2f((float)(e - ei)), k);
}

struct Smem {
  alignas(16) uint32_t xbuf[2][kTwCtas][8];  // exchanges: [round parity][source rank][words]
  alignas(8) uint64_t xbar[2];
  uint32_t mine[8];                         // this CTA's words of the current exchange
  int tok[kMaxNodes], first_child[kMaxNodes], next_sib[kMaxNodes];
  int path[kMaxNodes], out[kMaxNodes];
  float probe[kMaxNodes][4];
  int kids[kMaxNodes];
  double px[kMaxNodes], qx[kMaxNodes];  // per child of the node (position in kids)
  float gzt[kMaxNodes], gzd[kMaxNodes];
  double uk[kMaxNodes];  // accept uniform of each child of the node (position in kids)
  DecideCtx ctx;
  double invZ64[kMaxNodes + 1];
  dfloat wp[kTwCtas];                   // mass of p of the node per slice
  dfloat wr[kTwCtas];                   // mass of the last residual per slice
  Run rt[kTwWarps], rd[kTwWarps];
  float rz[kTwWarps];
  dfloat scan[kTwWarps];
  int nkids, node, a, child_i, accept, moved;
  int err, bad;
  int aT, aD;
  int owner, tok_out;
  float w_out;
  dfloat trel, Zdraw;
  int tile_hit, last_pos;
};

}  // namespace tw

// Exchange number `round` (every thread keeps the count): the CTA's 8 words
// (sh.mine, written before the call and followed by a __syncthreads) to
// slot [round & 1][rank] of every CTA, then the wait for the eight
// contributions to this CTA.  All threads call it; returns false everywhere
// if the wait gave up.  Two slots and two mbarriers alternate, so a CTA one
// exchange ahead of another never writes where the other still reads.
__device__ __forceinline__ bool tw_exchange(tw::Smem& sh, int rank, uint64_t limit, int& round) {
  const int par = round & 1;
  const int tid = threadIdx.x;
  if (tid < kTwCtas) {
    const uint32_t slot = ptx::smem_u32(&sh.xbuf[par][rank][0]);
    const uint32_t dst = tw::mapa(slot, (uint32_t)tid);
    tw::st_remote_v4(dst, sh.mine[0], sh.mine[1], sh.mine[2], sh.mine[3]);
    tw::st_remote_v4(dst + 16, sh.mine[4], sh.mine[5], sh.mine[6], sh.mine[7]);
    tw::arrive_remote(tw::mapa(ptx::smem_u32(&sh.xbar[par]), (uint32_t)tid));
  }
  if (tid == 0) {
    const uint32_t bar = ptx::smem_u32(&sh.xbar[par]);
    const uint32_t parity = (uint32_t)((round >> 1) & 1);
    bool ok = false;
    long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
      if (tw::try_wait_cluster(bar, parity)) {
        ok = true;
        break;
      }
      if ((it & 255u) == 255u) {
        const long long now = clock64();
        if (t0 == 0) {
          t0 = now;
        } else if ((uint64_t)(now - t0) > limit) {
          break;
        }
      }
    }
    if (!ok) sh.err = 1;
  }
  ++round;
  __syncthreads();
  return sh.err == 0;
}

// Block-wide: rows `trow` (and `drow` when non-null) of this CTA's slice
// [v0, v1) of 16-byte vectors -> each warp's runs in sh.rt[warp] /
// sh.rd[warp] (the caller merges the warps).
template <typename T>
__device__ void tw_slice_runs(const T* trow, const T* drow, int64_t v0, int64_t v1, float cs,
                              tw::Smem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  tw::Run rt{-INFINITY, 0.f, 0x7fffffff}, rd{-INFINITY, 0.f, 0x7fffffff};
  for (int64_t base = v0 + tid; base < v1; base += (int64_t)kTwThreads * kTwBatch) {
    uint4 xt[kTwBatch], xd[kTwBatch];
#pragma unroll
    for (int k = 0; k < kTwBatch; ++k) {
      const int64_t v = base + (int64_t)k * kTwThreads;
      xt[k] = v < v1 ? __ldg(reinterpret_cast<const uint4*>(trow) + v) : make_uint4(0, 0, 0, 0);
      xd[k] = (drow != nullptr && v < v1) ? __ldg(reinterpret_cast<const uint4*>(drow) + v)
                                          : make_uint4(0, 0, 0, 0);
    }
    // the batch: its maximum and first argmax, then its sum against that
    // maximum (independent terms), merged into the running values
    float ft[kTwBatch][EPV], fd[kTwBatch][EPV];
    tw::Run bt{-INFINITY, 0.f, 0x7fffffff}, bd{-INFINITY, 0.f, 0x7fffffff};
#pragma unroll
    for (int k = 0; k < kTwBatch; ++k) {
      const int64_t v = base + (int64_t)k * kTwThreads;
      unpack16(xt[k], ft[k]);
      unpack16(xd[k], fd[k]);
#pragma unroll
      for (int i = 0; i < EPV; ++i) {
        if (v >= v1) {
          ft[k][i] = -INFINITY;
          fd[k][i] = -INFINITY;
        }
        const int e = (int)(v * EPV + i);
        if (ft[k][i] > bt.m) {
          bt.m = ft[k][i];
          bt.a = e;
        }
        if (fd[k][i] > bd.m) {
          bd.m = fd[k][i];
          bd.a = e;
        }
      }
    }
    float st[2] = {0.f, 0.f}, sd[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kTwBatch; ++k)
#pragma unroll
      for (int i = 0; i < EPV; ++i) {
        if (ft[k][i] != -INFINITY) st[i & 1] += fast_exp2((ft[k][i] - bt.m) * cs);
        if (fd[k][i] != -INFINITY) sd[i & 1] += fast_exp2((fd[k][i] - bd.m) * cs);
      }
    bt.s = st[0] + st[1];
    bd.s = sd[0] + sd[1];
    rt = tw::run_merge(rt, bt, cs);
    if (drow != nullptr) rd = tw::run_merge(rd, bd, cs);
  }
  rt = tw::run_warp(rt, cs);
  rd = tw::run_warp(rd, cs);
  if (lane == 0) {
    sh.rt[warp] = rt;
    sh.rd[warp] = rd;
  }
  __syncthreads();
}

// Block-wide: this CTA's mass of the residual weights (nrej rejections so
// far) over its slice -- fp32 per thread and per warp, the warps combined by
// thread 0 in double-float -- left as this CTA's words in sh.mine.
template <typename T>
__device__ void tw_slice_mass(const T* trow, const T* drow, int64_t v0, int64_t v1,
                               const DecideCtx& c, int nrej, tw::Smem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  float s = 0.f;
  for (int64_t base = v0 + tid; base < v1; base += (int64_t)kTwThreads * kTwBatch) {
    uint4 xt[kTwBatch], xd[kTwBatch];
#pragma unroll
    for (int k = 0; k < kTwBatch; ++k) {
      const int64_t v = base + (int64_t)k * kTwThreads;
      xt[k] = v < v1 ? __ldg(reinterpret_cast<const uint4*>(trow) + v) : make_uint4(0, 0, 0, 0);
      xd[k] = v < v1 ? __ldg(reinterpret_cast<const uint4*>(drow) + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kTwBatch; ++k) {
      const int64_t v = base + (int64_t)k * kTwThreads;
      if (v >= v1) continue;
      float ft[EPV], fd[EPV];
      unpack16(xt[k], ft);
      unpack16(xd[k], fd);
      float s2[2] = {0.f, 0.f};
#pragma unroll
      for (int i = 0; i < EPV; ++i) s2[i & 1] += weight_plain(ft[i], fd[i], c, nrej);
      s += s2[0] + s2[1];
    }
  }
  s = warp_sum(s);
  if (lane == 0) sh.rz[warp] = s;
  __syncthreads();
  if (tid == 0) {  // the warps' sums in double-float: this CTA's words
    dfloat t = df_make(0.f);
    for (int w = 0; w < kTwWarps; ++w) t = df_add(t, df_make(sh.rz[w]));
    sh.mine[0] = __float_as_uint(t.hi);
    sh.mine[1] = __float_as_uint(t.lo);
  }
  __syncthreads();
}

// Block-wide inverse CDF inside this CTA's slice: the smallest element whose
// running weight (in index order, from the slice's start) exceeds sh.trel,
// else the last element of positive weight.  Thread 0 leaves the token and
// its weight in sh.tok_out / sh.w_out.
template <typename T>
__device__ void tw_slice_draw(const T* trow, const T* drow, int64_t v0, int64_t v1,
                              const DecideCtx& c, int nrej, tw::Smem& sh) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  dfloat rem = sh.trel;
  if (tid == 0) {
    sh.last_pos = -1;
    sh.tok_out = -1;
    sh.w_out = 0.f;
  }
  for (int64_t base = v0; base < v1; base += kTwThreads) {
    const int64_t v = base + tid;
    float w[EPV];
    float ts = 0.f;
    if (v < v1) {
      const uint4 xt = __ldg(reinterpret_cast<const uint4*>(trow) + v);
      const uint4 xd = nrej > 0 ? __ldg(reinterpret_cast<const uint4*>(drow) + v)
                                : make_uint4(0, 0, 0, 0);
      float ft[EPV], fd[EPV];
      unpack16(xt, ft);
      unpack16(xd, fd);
#pragma unroll
      for (int i = 0; i < EPV; ++i) {
        w[i] = weight_plain(ft[i], fd[i], c, nrej);
        ts += w[i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < EPV; ++i) w[i] = 0.f;
    }
    // inclusive scan of the threads' sums in index order (double-float)
    dfloat incl = df_warp_scan(df_make(ts));
    if (lane == kWarp - 1) sh.scan[warp] = incl;
    __syncthreads();
    dfloat wbase = df_make(0.f), total = df_make(0.f);
#pragma unroll
    for (int k = 0; k < kTwWarps; ++k) {
      if (k < warp) wbase = df_add(wbase, sh.scan[k]);
      total = df_add(total, sh.scan[k]);
    }
    incl = df_add(incl, wbase);
    const dfloat excl = df_sub(incl, df_make(ts));
    const bool hit = ts > 0.f && !df_gt(excl, rem) && df_gt(incl, rem);
    const unsigned hb = __ballot_sync(0xffffffffu, hit);
    const unsigned pb = __ballot_sync(0xffffffffu, ts > 0.f);
    if (tid == 0) sh.tile_hit = 0x7fffffff;
    __syncthreads();
    if (hb != 0 && lane == __ffs(hb) - 1) atomicMin(&sh.tile_hit, tid);
    if (pb != 0 && lane == 31 - __clz(pb)) atomicMax(&sh.last_pos, (int)(v * EPV));
    __syncthreads();
    const int ht = sh.tile_hit;
    if (ht != 0x7fffffff) {
      if (tid == ht) {
        dfloat cum = excl;
        int k = -1, klast = -1;
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
          if (w[i] > 0.f) {
            klast = i;
            cum = df_add(cum, df_make(w[i]));
            if (k < 0 && df_gt(cum, rem)) k = i;
          }
        }
        if (k < 0) k = klast;
        sh.tok_out = (int)(v * EPV + k);
        sh.w_out = w[k];
      }
      __syncthreads();
      return;
    }
    rem = df_sub(rem, total);
    __syncthreads();
  }
  // rounding at the very top: the last element of positive weight in the
  // slice (found by one more look at its last positive vector)
  if (tid == 0 && sh.last_pos >= 0) {
    const int64_t v = sh.last_pos / EPV;
    const uint4 xt = __ldg(reinterpret_cast<const uint4*>(trow) + v);
    const uint4 xd = nrej > 0 ? __ldg(reinterpret_cast<const uint4*>(drow) + v)
                              : make_uint4(0, 0, 0, 0);
    float ft[EPV], fd[EPV];
    unpack16(xt, ft);
    unpack16(xd, fd);
    for (int i = EPV - 1; i >= 0; --i) {
      const float wi = weight_plain(ft[i], fd[i], c, nrej);
      if (wi > 0.f) {
        sh.tok_out = (int)(v * EPV + i);
        sh.w_out = wi;
        break;
      }
    }
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kTwThreads) rs_tree_walk_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parent, const float* __restrict__ temperature, uint64_t seed,
    uint64_t offset, uint64_t b_base, int32_t* __restrict__ out_tokens, int32_t* __restrict__ path,
    int32_t* __restrict__ accepted_len, float* __restrict__ probe, spec_dims d, int n_chunks,
    const RowStat* stats, uint32_t* status, int inputs_ready) {
  constexpr int EPV = 16 / sizeof(T);
  __shared__ tw::Smem sh;
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const int rank = (int)tw::cluster_rank();
  const int b = blockIdx.x / kTwCtas;
  const int M = d.M, V = d.V;
  const uint64_t limit = wait_limit_cycles(d);
  int round = 0;  // exchanges so far (the same count in every thread)
  // Launched once everything before the statistics kernel has completed
  // (inputs_ready), the walk reads its inputs at once; otherwise (after the
  // LM heads) it waits for its predecessor first.
  if (!inputs_ready) pdl_wait();

  // ---- validation (every CTA alike) --------------------------------------
  const float temp = temperature[b];
  const bool greedy = temp == 0.f;
  const float cs = stat_scale(temp);
  if (tid == 0) {
    sh.bad = temperature_valid(temp) ? 0 : 1;
    sh.err = 0;
    sh.owner = -3;
    sh.tok_out = -1;
    sh.w_out = 0.f;
    sh.Zdraw = df_make(1.f);
    sh.moved = 0;
  }
  __syncthreads();
  for (int n = tid; n < M; n += kTwThreads) {
    const int32_t x = tokens[(int64_t)b * M + n];
    const int32_t pn = parent[(int64_t)b * M + n];
    sh.tok[n] = x;
    if (n == 0 ? pn != -1 : (pn < 0 || pn >= n)) atomicOr(&sh.bad, 1);
    if (n > 0 && (x < 0 || x >= V)) atomicOr(&sh.bad, 2);
    sh.out[n] = -1;
    sh.path[n] = -1;
    sh.probe[n][0] = sh.probe[n][1] = sh.probe[n][2] = sh.probe[n][3] = -1.f;
  }
  __syncthreads();
  if (sh.bad != 0) {
    if (rank == 0) {
      for (int n = tid; n < M; n += kTwThreads) {
        out_tokens[(int64_t)b * M + n] = -1;
        path[(int64_t)b * M + n] = -1;
        if (probe != nullptr)
          for (int k = 0; k < 4; ++k) probe[((int64_t)b * M + n) * 4 + k] = -1.f;
      }
      if (tid == 0) {
        accepted_len[b] = -1;
        raise_status(status, (sh.bad & 1) ? SPEC_ERR_INVALID_ARG : SPEC_ERR_DEVICE_BOUNDS);
      }
    }
    return;  // every CTA of the cluster leaves here alike
  }
  if (tid == 0) {
    for (int n = 0; n < M; ++n) sh.first_child[n] = -1;
    for (int n = M - 1; n >= 1; --n) {  // ascending sibling lists
      const int p = parent[(int64_t)b * M + n];
      sh.next_sib[n] = sh.first_child[p];
      sh.first_child[p] = n;
    }
    ptx::mbar_init(ptx::smem_u32(&sh.xbar[0]), kTwCtas);
    ptx::mbar_init(ptx::smem_u32(&sh.xbar[1]), kTwCtas);
    ptx::fence_mbar_init();
    sh.node = 0;
    sh.a = 0;
    sh.path[0] = 0;
  }
  const uint64_t bglob = b_base + (uint64_t)b;
  tw::cluster_sync();  // the mbarriers of every CTA are ready

  const int64_t NV = V / EPV;  // rows are whole 16-byte vectors
  const int64_t v0 = NV * rank / kTwCtas, v1 = NV * (rank + 1) / kTwCtas;
  const double cs64 = (double)cs;

  // ---- the walk ------------------------------------------------------------
  for (;;) {
    const int node = sh.node;
    const T* trow = target + ((int64_t)b * M + node) * V;
    const T* drow = draft + ((int64_t)b * M + node) * V;
    const bool has_kids = sh.first_child[node] >= 0;
    if (tid == 0) {
      int k = 0;
      for (int c = sh.first_child[node]; c >= 0; c = sh.next_sib[c]) sh.kids[k++] = c;
      sh.nkids = k;
    }
    __syncthreads();
    const int nk = sh.nkids;
    // the children's logits (every CTA alike), loaded with the slice
    T g_t = T(0.f), g_d = T(0.f);
    if (tid < nk) {
      const int64_t o = ((int64_t)b * M + node) * V + sh.tok[sh.kids[tid]];
      g_t = target[o];
      g_d = draft[o];
    }
    tw_slice_runs<T>(trow, has_kids ? drow : nullptr, v0, v1, cs, sh);
    if (tid < nk) {
      sh.gzt[tid] = to_f32(g_t);
      sh.gzd[tid] = to_f32(g_d);
    }
    if (tid == 0) {
      tw::Run rt = sh.rt[0], rd = sh.rd[0];
      for (int w = 1; w < kTwWarps; ++w) {
        rt = tw::run_merge(rt, sh.rt[w], cs);
        rd = tw::run_merge(rd, sh.rd[w], cs);
      }
      sh.mine[0] = __float_as_uint(rt.m);
      sh.mine[1] = __float_as_uint(rt.s);
      sh.mine[2] = (uint32_t)rt.a;
      sh.mine[3] = __float_as_uint(rd.m);
      sh.mine[4] = __float_as_uint(rd.s);
      sh.mine[5] = (uint32_t)rd.a;
      sh.mine[6] = 0u;
      sh.mine[7] = 0u;
    }
    __syncthreads();
    if (!tw_exchange(sh, rank, limit, round)) break;
    const int par = (round - 1) & 1;
    if (warp == 0) {
      // the node's normalisers from the slices: lane r < kTwCtas holds
      // slice r; the same shuffles in every CTA give the same values
      const bool live = lane < kTwCtas;
      const uint32_t* x = sh.xbuf[par][live ? lane : 0];
      const float mr = live ? __uint_as_float(x[0]) : -INFINITY;
      const float sr = live ? __uint_as_float(x[1]) : 0.f;
      const float mdr = live ? __uint_as_float(x[3]) : -INFINITY;
      const float sdr = live ? __uint_as_float(x[4]) : 0.f;
      const float mT = warp_max(mr), mD = warp_max(mdr);
      const dfloat wt = mr == -INFINITY ? df_make(0.f)
                                        : df_mul_f(df_make(sr), fast_exp2((mr - mT) * cs));
      const dfloat wd = mdr == -INFINITY ? df_make(0.f)
                                         : df_mul_f(df_make(sdr), fast_exp2((mdr - mD) * cs));
      const dfloat sT = df_warp_sum(wt), sD = df_warp_sum(wd);
      // the first slice (lowest indices) holding the maximum gives the argmax
      const unsigned ht = __ballot_sync(0xffffffffu, live && mr == mT);
      const unsigned hd = __ballot_sync(0xffffffffu, live && mdr == mD);
      const int aT = __shfl_sync(0xffffffffu, live ? (int)x[2] : 0, ht ? __ffs(ht) - 1 : 0);
      const int aD = __shfl_sync(0xffffffffu, live ? (int)x[5] : 0, hd ? __ffs(hd) - 1 : 0);
      if (live) {
        sh.wp[lane] = wt;
        sh.wr[lane] = df_make(0.f);
      }
      // the children's P(x), Q(x) and accept uniforms (counter word 0: the
      // child's node index + 1), one child a lane; the row sums' reciprocals
      // meanwhile on the last two lanes (fp64 is slow here: its dependent
      // chains are kept short and side by side)
      double inv = 0.0;
      if (lane == kWarp - 1) inv = 1.0 / df_to_d(sT);
      if (lane == kWarp - 2) inv = has_kids ? 1.0 / df_to_d(sD) : 0.0;
      const double invST = __shfl_sync(0xffffffffu, inv, kWarp - 1);
      const double invSD = __shfl_sync(0xffffffffu, inv, kWarp - 2);
      for (int i = lane; i < nk; i += kWarp) {
        const int x = sh.tok[sh.kids[i]];
        if (greedy) {
          sh.px[i] = x == aT ? 1.0 : 0.0;
          sh.qx[i] = x == aD ? 1.0 : 0.0;
        } else {
          const double et = ((double)sh.gzt[i] - (double)mT) * cs64;
          const double ed = ((double)sh.gzd[i] - (double)mD) * cs64;
          sh.px[i] = tw::exp2_split(et) * invST;
          sh.qx[i] = tw::exp2_split(ed) * invSD;
          const Philox4 r = philox4x64_10((uint64_t)sh.kids[i] + 1, bglob, offset, 0, seed, 0);
          sh.uk[i] = (double)u24(r.w[0]);
        }
      }
      if (lane == 0) {
        sh.aT = ht == 0 || aT < 0 || aT >= V ? 0 : aT;
        sh.aD = hd == 0 || aD < 0 || aD >= V ? 0 : aD;
        ctx_no_filter(sh.ctx);
        sh.ctx.mT = mT;
        sh.ctx.invST = (float)invST;
        sh.ctx.cs = cs;
        sh.ctx.nrej = 0;
        sh.ctx.mD = has_kids ? mD : 0.f;
        sh.ctx.invSD = has_kids ? (float)invSD : 0.f;
        sh.invZ64[0] = 1.0;
        sh.child_i = 0;
        sh.moved = 0;
      }
    }
    __syncthreads();
    // ---- the children in order ---------------------------------------------
    while (sh.child_i < nk) {
      const int i = sh.child_i;
      const int c = sh.kids[i];
      if (tid == 0) {
        bool acc;
        if (greedy) {
          acc = sh.px[i] > 0.0;
          sh.probe[c][0] = (float)sh.px[i];
          sh.probe[c][1] = (float)sh.qx[i];
        } else {
          const double Q = sh.qx[i];
          double P = sh.px[i];
          for (int j = 1; j <= sh.ctx.nrej; ++j) P = fmax(P - Q, 0.0) * sh.invZ64[j];
          acc = sh.uk[i] * Q < P;
          sh.probe[c][0] = (float)P;
          sh.probe[c][1] = (float)Q;
        }
        sh.accept = acc;
        sh.moved = acc;
      }
      __syncthreads();
      if (sh.accept) break;
      if (!greedy) {
        // the residual after this rejection: its mass over the slices
        const int nrej_next = sh.ctx.nrej + 1;
        tw_slice_mass<T>(trow, drow, v0, v1, sh.ctx, nrej_next, sh);
        if (!tw_exchange(sh, rank, limit, round)) break;
        if (warp == 0) {
          const int p2 = (round - 1) & 1;
          const bool live = lane < kTwCtas;
          const dfloat zr = live ? dfloat{__uint_as_float(sh.xbuf[p2][lane][0]),
                                          __uint_as_float(sh.xbuf[p2][lane][1])}
                                 : df_make(0.f);
          const dfloat Zd = df_warp_sum(zr);
          if (live) sh.wr[lane] = zr;
          if (lane == 0) {
            const double Z = df_to_d(Zd);
            if (Z > 0.0) {
              const int j = nrej_next;
              sh.ctx.nrej = j;
              sh.ctx.Z[j] = Z;
              sh.invZ64[j] = 1.0 / Z;
              sh.ctx.invZ[j] = (float)sh.invZ64[j];
            } else {
              // a residual of zero mass: back to p of the node
              sh.ctx.nrej = 0;
            }
          }
        }
      }
      if (tid == 0) sh.child_i = i + 1;
      __syncthreads();
    }
    if (sh.err != 0) break;
    if (sh.moved) {
      if (tid == 0) {
        const int c = sh.kids[sh.child_i];
        const int a = sh.a + 1;
        sh.a = a;
        sh.path[a] = c;
        sh.out[a - 1] = sh.tok[c];
        sh.node = c;
      }
      __syncthreads();
      continue;
    }
    // ---- the draw at `node` --------------------------------------------------
    if (greedy) {
      if (tid == 0) {
        sh.owner = -1;
        sh.tok_out = sh.aT;
        sh.w_out = 1.f;
        sh.Zdraw = df_make(1.f);
        sh.probe[node][2] = 1.f;
        sh.probe[node][3] = 1.f;
      }
      __syncthreads();
      break;
    }
    if (warp == 0) {
      // the slice holding u * Z: the first of positive mass whose running
      // mass (in rank order) exceeds it, else the last of positive mass
      const int nrej = sh.ctx.nrej;
      const bool live = lane < kTwCtas;
      const dfloat w = live ? (nrej > 0 ? sh.wr[lane] : sh.wp[lane]) : df_make(0.f);
      const dfloat incl = df_warp_scan(w);
      const dfloat Z = df_shfl(incl, kWarp - 1);
      const Philox4 r = philox4x64_10((uint64_t)node + 1, bglob, offset, 0, seed, 0);
      const dfloat t = df_mul_f(Z, u24(r.w[1]));
      const bool pos = live && w.hi > 0.f;
      const unsigned hit = __ballot_sync(0xffffffffu, pos && df_gt(incl, t));
      const unsigned pb = __ballot_sync(0xffffffffu, pos);
      const int owner = hit ? __ffs(hit) - 1 : (pb ? 31 - __clz(pb) : 0);
      const dfloat excl = df_shfl(df_sub(incl, w), owner);
      if (lane == 0) {
        sh.owner = owner;
        sh.trel = df_sub(t, excl);
        sh.Zdraw = Z;
        sh.probe[node][2] = nrej > 0 ? (float)sh.ctx.Z[nrej] : 1.f;
      }
    }
    __syncthreads();
    if (sh.owner == rank) tw_slice_draw<T>(trow, drow, v0, v1, sh.ctx, sh.ctx.nrej, sh);
    break;
  }
  pdl_trigger();

  // ---- the verdict: every row the request needs has a distribution -------
  pdl_wait();  // the statistics pass has completed
  int bad_rows = 0;
  const bool stats_lost = (ld_volatile_u32(status) >> SPEC_ERR_TIMEOUT) & 1u;
  if (!stats_lost) {
    for (int k = rank + kTwCtas * warp; k < 2 * M; k += kTwCtas * kTwWarps) {
      const int which = k / M, n = k % M;
      if (which == 1 && sh.first_child[n] < 0) continue;
      const RowStat* st = stats + (((int64_t)b * 2 + which) * M + n) * n_chunks;
      float m = -INFINITY;
      for (int c = lane; c < n_chunks; c += kWarp) m = fmaxf(m, ld_stat_cg(st + c).m);
      m = warp_max(m);
      float s = 0.f;
      for (int c = lane; c < n_chunks; c += kWarp) {
        const RowStat x = ld_stat_cg(st + c);
        if (x.m != -INFINITY) s += (float)x.s * fast_exp2((x.m - m) * cs);
      }
      s = warp_sum(s);
      bad_rows |= !(m > -INFINITY && m < INFINITY && s > 0.f && s < INFINITY);
    }
  }
  bad_rows = __syncthreads_or(bad_rows);
  if (tid == 0) {
    sh.mine[0] = (uint32_t)(bad_rows | (stats_lost ? 2 : 0) | (sh.err ? 4 : 0));
    sh.mine[1] = (uint32_t)(sh.owner == rank ? sh.tok_out : -1);
    sh.mine[2] = __float_as_uint(sh.owner == rank ? sh.w_out : 0.f);
  }
  __syncthreads();
  const bool ok = tw_exchange(sh, rank, limit, round);
  if (tid == 0 && sh.err) raise_status(status, SPEC_ERR_TIMEOUT);
  if (rank == 0) {
    const int p2 = (round - 1) & 1;
    int flags = ok ? 0 : 4;
    int tok = sh.owner == -1 ? sh.tok_out : -1;  // temperature 0: every CTA knows it
    float wtok = sh.owner == -1 ? sh.w_out : 0.f;
    for (int r = 0; r < kTwCtas; ++r) {
      flags |= (int)sh.xbuf[p2][r][0];
      if (r == sh.owner) {
        tok = (int)sh.xbuf[p2][r][1];
        wtok = __uint_as_float(sh.xbuf[p2][r][2]);
      }
    }
    const bool fail = flags != 0 || tok < 0 || tok >= V;
    const int a = sh.a;
    for (int n = tid; n < M; n += kTwThreads) {
      int o = fail ? -1 : sh.out[n];
      if (!fail && n == a) o = tok;
      out_tokens[(int64_t)b * M + n] = o;
      path[(int64_t)b * M + n] = fail ? -1 : sh.path[n];
      if (probe != nullptr) {
        float pv[4] = {sh.probe[n][0], sh.probe[n][1], sh.probe[n][2], sh.probe[n][3]};
        if (!fail && n == sh.node && !greedy) pv[3] = wtok / df_to_f(sh.Zdraw);
        for (int k = 0; k < 4; ++k) probe[((int64_t)b * M + n) * 4 + k] = fail ? -1.f : pv[k];
      }
    }
    if (tid == 0) {
      accepted_len[b] = fail ? -1 : a;
      if (flags & 4) raise_status(status, SPEC_ERR_TIMEOUT);
      else if (flags & 1) raise_status(status, SPEC_ERR_NONFINITE);
      else if (fail && !(flags & 2)) raise_status(status, SPEC_ERR_NONFINITE);
      // (flags & 2: the statistics pass gave up and raised the time-out)
    }
  }
  tw::cluster_sync();  // no CTA leaves while another may still write to it
}

bool rs_tree_walk_supported(const spec_dims& d, bool aligned, bool tree, bool filters) {
  return aligned && tree && !filters && d.M >= 1 && d.M <= kMaxNodes;
}

template <typename T>
static cudaError_t launch_tw(const RsArgs& a, const WsLayout& lay, bool inputs_ready,
                             cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kTwCtas;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.d.B * kTwCtas));
  cfg.blockDim = dim3(kTwThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  char* ws = static_cast<char*>(a.ws);
  return cudaLaunchKernelEx(&cfg, rs_tree_walk_kernel<T>, static_cast<const T*>(a.target),
                            static_cast<const T*>(a.draft), a.tokens, a.parent, a.temperature,
                            a.seed, a.offset, a.b_base, a.out_tokens, a.path, a.accepted_len,
                            a.probe, a.d, lay.rs_chunks,
                            (const RowStat*)reinterpret_cast<RowStat*>(ws + lay.rs_off),
                            reinterpret_cast<uint32_t*>(ws + lay.status_off),
                            inputs_ready ? 1 : 0);
}

cudaError_t rs_tree_walk_launch(const RsArgs& a, const WsLayout& lay, bool inputs_ready,
                                cudaStream_t st) {
  return a.d.logits_dtype == SPEC_BF16 ? launch_tw<__nv_bfloat16>(a, lay, inputs_ready, st)
                                       : launch_tw<float>(a, lay, inputs_ready, st);
}

}  // namespace specv
