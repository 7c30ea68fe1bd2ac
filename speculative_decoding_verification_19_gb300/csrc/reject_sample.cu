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
// Two kernels:
//   rs_rowstats_kernel  one CTA per (chunk of 8192 logits, row, request):
//                       chunk max m_c and s_c = sum exp2((z - m_c)*log2e/T)
//                       (fp32 terms, fp64 sums), over every target row and
//                       every draft row that drafted children.  This is the
//                       HBM-streaming pass: each logit is read once, with
//                       16-byte coalesced loads.
//   rs_decide_kernel    one CTA per request: merges the chunk statistics into
//                       row normalisers (fp64), runs the sequential accept
//                       tests in fp64, and draws the replacement/bonus token
//                       with a two-level inverse CDF (per-sweep sums, then a
//                       block scan inside the selected sweep).
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "philox.cuh"
#include "reject_sample.cuh"

namespace specv {

constexpr int kRsThreads = 256;   // rowstats CTA size
constexpr int kRsVecs = 4;        // 16-byte vectors per thread per chunk
constexpr int kDecThreads = 512;  // decide CTA size
constexpr int kDecWarps = kDecThreads / kWarp;
constexpr int kMaxM = 64;
constexpr int kMaxSweeps = 256;

int rs_chunk_elems(int logits_dtype) {
  return kRsThreads * kRsVecs * (logits_dtype == SPEC_BF16 ? 8 : 4);
}
int rs_max_vocab(int logits_dtype) {
  return kMaxSweeps * kDecThreads * (logits_dtype == SPEC_BF16 ? 8 : 4);
}

__device__ __forceinline__ bool temperature_ok(float T) {
  return T >= FLT_MIN && T <= FLT_MAX;  // normal, positive, finite (NaN fails)
}

// Load EPV consecutive logits starting at element e (-inf past the row end).
template <typename T, bool kAligned>
__device__ __forceinline__ void load_vec(const T* row, int64_t e, int V, float (&f)[16 / sizeof(T)]) {
  constexpr int EPV = 16 / sizeof(T);
  if (kAligned && e + EPV <= V) {
    const uint4 r = __ldg(reinterpret_cast<const uint4*>(row + e));
    unpack16(r, f);
  } else {
#pragma unroll
    for (int i = 0; i < EPV; ++i) f[i] = (e + i < V) ? to_f32(row[e + i]) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// pass 1: chunk statistics
// ---------------------------------------------------------------------------
template <typename T, bool kAligned>
__global__ void __launch_bounds__(kRsThreads) rs_rowstats_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ parent,
    const float* __restrict__ temperature, spec_dims d, int n_chunks, RowStat* __restrict__ stats) {
  constexpr int EPV = 16 / sizeof(T);
  // flat task index over (request, row, chunk), chunks fastest
  const int64_t task = blockIdx.x;
  const int c = (int)(task % n_chunks);
  const int row = (int)((task / n_chunks) % (2 * d.M));
  const int b = (int)(task / ((int64_t)n_chunks * 2 * d.M));
  const int which = row / d.M, n = row % d.M;
  const int tid = threadIdx.x;
  if (which == 1) {  // a draft row is read only if its node drafted children
    int has_child;
    if (parent == nullptr) {
      has_child = n < d.M - 1;
    } else {
      const int k = n + 1 + tid;
      has_child = __syncthreads_or(k < d.M && parent[(int64_t)b * d.M + k] == n);
    }
    if (!has_child) return;
  }
  const float temp = temperature[b];
  const float cs = temperature_ok(temp) ? 1.4426950408889634f / temp : 1.0f;
  const T* rowp = (which == 0 ? target : draft) + ((int64_t)b * d.M + n) * d.V;
  const int64_t e0 = (int64_t)c * (kRsThreads * kRsVecs * EPV);

  float f[kRsVecs][EPV];
  float mt = -INFINITY;
#pragma unroll
  for (int v = 0; v < kRsVecs; ++v) {
    load_vec<T, kAligned>(rowp, e0 + ((int64_t)v * kRsThreads + tid) * EPV, d.V, f[v]);
#pragma unroll
    for (int i = 0; i < EPV; ++i) mt = fmaxf(mt, f[v][i]);
  }
  __shared__ float s_max[kRsThreads / kWarp];
  __shared__ double s_sum[kRsThreads / kWarp];
  mt = warp_max(mt);
  if (tid % kWarp == 0) s_max[tid / kWarp] = mt;
  __syncthreads();
  float mc = s_max[0];
#pragma unroll
  for (int w = 1; w < kRsThreads / kWarp; ++w) mc = fmaxf(mc, s_max[w]);
  float st = 0.f;
  if (mc != -INFINITY) {
#pragma unroll
    for (int v = 0; v < kRsVecs; ++v)
#pragma unroll
      for (int i = 0; i < EPV; ++i) st += fast_exp2((f[v][i] - mc) * cs);
  }
  double sd = warp_sum((double)st);
  if (tid % kWarp == 0) s_sum[tid / kWarp] = sd;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
#pragma unroll
    for (int w = 0; w < kRsThreads / kWarp; ++w) s += s_sum[w];
    RowStat r;
    r.m = mc;
    r.pad = 0.f;
    r.s = s;
    stats[(((int64_t)b * 2 + which) * d.M + n) * n_chunks + c] = r;
  }
}

// ---------------------------------------------------------------------------
// pass 2: decisions and the draw
// ---------------------------------------------------------------------------
struct DecideCtx {
  float mT, mD;       // row maxima of the node's target / draft rows
  float invST, invSD; // 1 / row sums (fp32)
  float cs;           // log2(e) / T
  int nrej;           // rejections so far at this node (working P = P_nrej)
  float invZ[kMaxM];  // 1 / Z_j of the residuals taken so far (element path)
  double Z[kMaxM];    // Z_j in fp64 (accept-test path)
};

// Weight of element e of the node's sampling / residual law:
//   nrej == 0:  exp2((z - mT) * cs)                     (unnormalised p)
//   nrej >= 1:  max(0, P_{nrej-1} - q)                  (unnormalised residual)
// with P_0 = p and P_j = max(0, P_{j-1} - q) / Z_j.
__device__ __forceinline__ float weight_of(float zt, float zd, const DecideCtx& c, int nrej) {
  const float et = fast_exp2((zt - c.mT) * c.cs);
  if (nrej == 0) return et;
  const float qv = fast_exp2((zd - c.mD) * c.cs) * c.invSD;
  float P = et * c.invST;
  for (int j = 1; j < nrej; ++j) P = fmaxf(P - qv, 0.f) * c.invZ[j];
  return fmaxf(P - qv, 0.f);
}

template <typename T, bool kAligned>
__device__ __forceinline__ float vec_weights(const T* trow, const T* drow, int64_t e, int V,
                                             const DecideCtx& c, int nrej,
                                             float (&w)[16 / sizeof(T)]) {
  constexpr int EPV = 16 / sizeof(T);
  float zt[EPV], zd[EPV];
  load_vec<T, kAligned>(trow, e, V, zt);
  if (nrej > 0) {
    load_vec<T, kAligned>(drow, e, V, zd);
  } else {
#pragma unroll
    for (int i = 0; i < EPV; ++i) zd[i] = 0.f;
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPV; ++i) {
    w[i] = (e + i < V) ? weight_of(zt[i], zd[i], c, nrej) : 0.f;
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

template <typename T, bool kAligned>
__global__ void __launch_bounds__(kDecThreads) rs_decide_kernel(
    const T* __restrict__ target, const T* __restrict__ draft, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parent, const float* __restrict__ temperature, uint64_t seed,
    uint64_t offset, uint64_t b_base, int32_t* __restrict__ out_tokens, int32_t* __restrict__ path,
    int32_t* __restrict__ accepted_len, float* __restrict__ probe, spec_dims d, int n_chunks,
    const RowStat* __restrict__ stats, uint32_t* __restrict__ status) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kSweep = kDecThreads * EPV;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int warp = tid / kWarp, lane = tid % kWarp;
  const int M = d.M, V = d.V;

  __shared__ int first_child[kMaxM], next_sib[kMaxM], tok[kMaxM];
  __shared__ float rowM[2][kMaxM];
  __shared__ double rowS[2][kMaxM];
  __shared__ double red[kDecWarps];
  __shared__ double warp_part[kMaxSweeps][kDecWarps];
  __shared__ double sweep_sum[kMaxSweeps];
  __shared__ DecideCtx ctx;
  __shared__ int s_node, s_child, s_accept, s_sweep, s_claim, s_a;
  __shared__ double s_t;

  // defined outputs first
  for (int i = tid; i < M; i += kDecThreads) {
    out_tokens[(int64_t)b * M + i] = -1;
    path[(int64_t)b * M + i] = -1;
  }
  if (probe != nullptr)
    for (int i = tid; i < 4 * M; i += kDecThreads) probe[(int64_t)b * M * 4 + i] = -1.f;

  // ---- validation --------------------------------------------------------
  const float temp = temperature[b];
  int bad_arg = !temperature_ok(temp);
  int bad_tok = 0;
  if (tid < M) {
    const int32_t x = tokens[(int64_t)b * M + tid];
    tok[tid] = x;
    if (tid > 0) bad_tok = (x < 0 || x >= V);
    if (parent != nullptr) {
      const int32_t pn = parent[(int64_t)b * M + tid];
      bad_arg |= (tid == 0) ? (pn != -1) : (pn < 0 || pn >= tid);
    }
  }
  bad_arg = __syncthreads_or(bad_arg);
  bad_tok = __syncthreads_or(bad_tok);
  if (tid == 0 && !bad_arg) {
    for (int n = 0; n < M; ++n) first_child[n] = -1;
    for (int n = M - 1; n >= 1; --n) {  // ascending sibling lists
      const int p = parent ? parent[(int64_t)b * M + n] : n - 1;
      next_sib[n] = first_child[p];
      first_child[p] = n;
    }
  }
  __syncthreads();
  const float cs = temperature_ok(temp) ? 1.4426950408889634f / temp : 1.0f;

  // ---- row normalisers ---------------------------------------------------
  int bad_row = 0;
  if (!bad_arg) {
    for (int r = warp; r < 2 * M; r += kDecWarps) {
      const int which = r / M, n = r % M;
      if (which == 1 && first_child[n] < 0) continue;
      const RowStat* st = stats + (((int64_t)b * 2 + which) * M + n) * n_chunks;
      float m = -INFINITY;
      for (int c = lane; c < n_chunks; c += kWarp) m = fmaxf(m, st[c].m);
      m = warp_max(m);
      double s = 0.0;
      for (int c = lane; c < n_chunks; c += kWarp) {
        const RowStat x = st[c];
        s += x.s * (double)exp2f((x.m - m) * cs);
      }
      s = warp_sum(s);
      if (lane == 0) {
        rowM[which][n] = m;
        rowS[which][n] = s;
      }
      bad_row |= !(m > -INFINITY && m < INFINITY && s > 0.0 && s < INFINITY);
    }
  }
  bad_row = __syncthreads_or(bad_row);
  if (bad_arg || bad_tok || bad_row) {
    if (tid == 0) {
      accepted_len[b] = -1;
      raise_status(status, bad_arg ? SPEC_ERR_INVALID_ARG
                           : bad_tok ? SPEC_ERR_DEVICE_BOUNDS
                                     : SPEC_ERR_NONFINITE);
    }
    return;
  }

  // ---- the walk ----------------------------------------------------------
  const uint64_t bglob = b_base + (uint64_t)b;
  const double cs64 = (double)cs;
  if (tid == 0) {
    s_node = 0;
    s_a = 0;
    path[(int64_t)b * M] = 0;
  }
  for (;;) {
    __syncthreads();
    const int node = s_node;
    const T* trow = target + ((int64_t)b * M + node) * V;
    const T* drow = draft + ((int64_t)b * M + node) * V;
    if (tid == 0) {
      ctx.mT = rowM[0][node];
      ctx.invST = (float)(1.0 / rowS[0][node]);
      ctx.cs = cs;
      ctx.nrej = 0;
      if (first_child[node] >= 0) {
        ctx.mD = rowM[1][node];
        ctx.invSD = (float)(1.0 / rowS[1][node]);
      } else {
        ctx.mD = 0.f;
        ctx.invSD = 0.f;
      }
      s_child = first_child[node];
    }
    __syncthreads();
    bool moved = false;
    while (s_child >= 0) {
      const int child = s_child;
      if (tid == 0) {
        // accept test of `child` in fp64
        const int x = tok[child];
        const double zt = (double)to_f32(trow[x]);
        const double zd = (double)to_f32(drow[x]);
        const double Q = exp2((zd - (double)ctx.mD) * cs64) / rowS[1][node];
        double P = exp2((zt - (double)ctx.mT) * cs64) / rowS[0][node];
        for (int j = 1; j <= ctx.nrej; ++j) P = fmax(P - Q, 0.0) / ctx.Z[j];
        const Philox4 r = philox4x64_10((uint64_t)child + 1, bglob, offset, 0, seed, 0);
        const double u = (double)u24(r.w[0]);
        s_accept = (u * Q < P);
        if (probe != nullptr) {
          probe[((int64_t)b * M + child) * 4 + 0] = (float)P;
          probe[((int64_t)b * M + child) * 4 + 1] = (float)Q;
        }
      }
      __syncthreads();
      if (s_accept) {
        moved = true;
        break;
      }
      const bool more = next_sib[child] >= 0;
      if (more) {
        // mass of the next residual, needed by the next sibling's test
        const int nrej_next = ctx.nrej + 1;
        double acc = 0.0;
        for (int64_t e = (int64_t)tid * EPV; e < V; e += kSweep) {
          float w[EPV];
          acc += (double)vec_weights<T, kAligned>(trow, drow, e, V, ctx, nrej_next, w);
        }
        const double Z = block_sum(acc, red);
        if (tid == 0) {
          if (Z > 0.0) {
            ctx.nrej = ctx.nrej + 1;
            ctx.invZ[ctx.nrej] = (float)(1.0 / Z);
            ctx.Z[ctx.nrej] = Z;
          } else {
            ctx.nrej = 0;  // zero-mass residual: fall back to p of the node
          }
        }
      } else if (tid == 0) {
        ctx.nrej = ctx.nrej + 1;
      }
      if (tid == 0) s_child = next_sib[child];
      __syncthreads();
    }
    if (moved) {
      if (tid == 0) {
        const int child = s_child;
        const int a = s_a + 1;
        s_a = a;
        path[(int64_t)b * M + a] = child;
        out_tokens[(int64_t)b * M + a - 1] = tok[child];
        s_node = child;
      }
      continue;
    }

    // ---- draw at `node` from the working law (inverse CDF) ---------------
    const Philox4 r = philox4x64_10((uint64_t)node + 1, bglob, offset, 0, seed, 0);
    const double u = (double)u24(r.w[1]);
    const int n_sweeps = ceil_div(V, kSweep);
    for (int attempt = 0; attempt < 2; ++attempt) {
      __syncthreads();
      const int nrej_now = ctx.nrej;
      for (int s = 0; s < n_sweeps; ++s) {
        float w[EPV];
        const float vs = vec_weights<T, kAligned>(trow, drow, (int64_t)s * kSweep + (int64_t)tid * EPV,
                                                  V, ctx, nrej_now, w);
        const double ws = warp_sum((double)vs);
        if (lane == 0) warp_part[s][warp] = ws;
      }
      __syncthreads();
      for (int s = tid; s < n_sweeps; s += kDecThreads) {
        double t = 0.0;
#pragma unroll
        for (int i = 0; i < kDecWarps; ++i) t += warp_part[s][i];
        sweep_sum[s] = t;
      }
      __syncthreads();
      if (tid == 0) {
        double Z = 0.0;
        for (int s = 0; s < n_sweeps; ++s) Z += sweep_sum[s];
        s_t = Z;
      }
      __syncthreads();
      if (s_t > 0.0 || attempt == 1) break;
      if (tid == 0) ctx.nrej = 0;  // zero-mass residual: draw from p of the node
    }
    if (tid == 0) {
      const double Z = s_t;
      const double t = u * Z;
      double pre = 0.0;
      int sel = -1, last_pos = 0;
      for (int s = 0; s < n_sweeps; ++s) {
        if (sweep_sum[s] > 0.0) last_pos = s;
        if (sel < 0 && pre + sweep_sum[s] > t) {
          sel = s;
          break;
        }
        pre += sweep_sum[s];
      }
      if (sel < 0) {  // rounding at the very top: take the last non-empty sweep
        sel = last_pos;
        pre = 0.0;
        for (int s = 0; s < sel; ++s) pre += sweep_sum[s];
      }
      s_sweep = sel;
      red[0] = t - pre;  // target inside the sweep
      red[1] = Z;
      s_claim = kDecThreads;
    }
    __syncthreads();
    const double trel = red[0];
    const double Ztot = red[1];
    // block exclusive scan of the per-thread vector sums of the selected sweep
    const int nrej_fin = ctx.nrej;
    const int64_t e = (int64_t)s_sweep * kSweep + (int64_t)tid * EPV;
    float w[EPV];
    const double vs = (double)vec_weights<T, kAligned>(trow, drow, e, V, ctx, nrej_fin, w);
    double incl = vs;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __shared__ double wtot[kDecWarps];
    __shared__ int last_nonzero;
    if (lane == kWarp - 1) wtot[warp] = incl;
    if (tid == 0) last_nonzero = -1;
    __syncthreads();
    double wpre = 0.0;
    for (int i = 0; i < warp; ++i) wpre += wtot[i];
    const double excl = wpre + incl - vs;
    if (vs > 0.0) atomicMax(&last_nonzero, tid);
    if (vs > 0.0 && excl <= trel && trel < excl + vs) atomicMin(&s_claim, tid);
    __syncthreads();
    int owner = s_claim;
    if (owner == kDecThreads) owner = last_nonzero;  // rounding gap: take the last mass
    if (owner < 0) owner = 0;
    if (tid == owner) {
      double cum = excl;
      int k = -1, lastpos = -1;
      for (int i = 0; i < EPV; ++i) {
        if (w[i] > 0.f) lastpos = i;
        cum += (double)w[i];
        if (k < 0 && cum > trel) k = i;
      }
      if (k < 0 || w[k] <= 0.f) k = lastpos;
      if (k < 0) k = 0;
      const int token = (int)(e + k);
      const int a = s_a;
      out_tokens[(int64_t)b * M + a] = token;
      accepted_len[b] = a;
      if (probe != nullptr) {
        probe[((int64_t)b * M + node) * 4 + 2] = nrej_fin == 0 ? 1.0f : (float)Ztot;
        probe[((int64_t)b * M + node) * 4 + 3] = (float)((double)w[k] / Ztot);
      }
    }
    return;
  }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
template <typename T, bool kAligned>
static cudaError_t launch_rs_t(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  const spec_dims& d = a.d;
  RowStat* stats = reinterpret_cast<RowStat*>(static_cast<char*>(a.ws) + lay.rs_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<char*>(a.ws) + lay.status_off);
  const unsigned g1 = (unsigned)((int64_t)lay.rs_chunks * 2 * d.M * d.B);
  rs_rowstats_kernel<T, kAligned><<<g1, kRsThreads, 0, st>>>(
      static_cast<const T*>(a.target), static_cast<const T*>(a.draft), a.parent, a.temperature, d,
      lay.rs_chunks, stats);
  ++*launches;
  rs_decide_kernel<T, kAligned><<<d.B, kDecThreads, 0, st>>>(
      static_cast<const T*>(a.target), static_cast<const T*>(a.draft), a.tokens, a.parent,
      a.temperature, a.seed, a.offset, a.b_base, a.out_tokens, a.path, a.accepted_len, a.probe, d,
      lay.rs_chunks, stats, status);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t rs_launch(const RsArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  const int esz = a.d.logits_dtype == SPEC_BF16 ? 2 : 4;
  const bool aligned = ((size_t)a.d.V * esz) % 16 == 0 &&
                       (reinterpret_cast<uintptr_t>(a.target) % 16) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.draft) % 16) == 0;
  if (a.d.logits_dtype == SPEC_BF16)
    return aligned ? launch_rs_t<__nv_bfloat16, true>(a, lay, st, launches)
                   : launch_rs_t<__nv_bfloat16, false>(a, lay, st, launches);
  return aligned ? launch_rs_t<float, true>(a, lay, st, launches)
                 : launch_rs_t<float, false>(a, lay, st, launches);
}

}  // namespace specv
