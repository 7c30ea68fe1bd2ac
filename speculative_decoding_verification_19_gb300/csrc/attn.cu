// KV append and verify attention over a paged KV cache.
//
// What is computed (page 1 §2.1, page 2 §3.3, page 3 tree-attention
// section): the M new rows of each request (pending root + drafts, or tree
// nodes) have their K/V appended at positions ctx..ctx+M-1; row i then
// attends to the cached prefix 0..ctx-1 and to the new positions of its
// ancestors and itself, which makes the one-pass result equal to
// token-by-token decoding.
//
// Kernels in this file (CUDA cores; the tensor-core path lives in
// attn_tc.cu):
//   kv_append_kernel   one CTA per request: checks the request (capacity,
//                      block ids, topology), records the verdict, writes the
//                      new K/V and clears the rest of the last block.
//   attn_split_kernel  split-KV attention: one CTA per (request, KV head,
//                      key range); all group*M query rows that read the KV
//                      head are handled together, so every K/V byte is read
//                      once per range.  Online softmax in base 2.
//   attn_combine_kernel  merges the per-range partials by log-sum-exp.
#include <math.h>

#include "attn.cuh"
#include "common.cuh"

namespace specv {

// ---------------------------------------------------------------------------
// append + per-request verdict
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) kv_append_kernel(
    const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ k_cache,
    T* __restrict__ v_cache, const int32_t* __restrict__ block_table,
    const int32_t* ctx_lens, const int32_t* __restrict__ parent, spec_dims d,
    int32_t* __restrict__ req_ok, uint32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // the inputs and the cache may come from the previous kernel
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int ctx = ctx_lens[b];
  const int64_t L = (int64_t)ctx + d.M;
  const int64_t cap = (int64_t)d.max_blocks * kBlock;
  const int32_t* bt = block_table + (int64_t)b * d.max_blocks;

  // capacity
  const bool cap_ok = ctx >= 0 && L <= cap;
  // block ids of every page the request reads or writes
  int bad_block = 0;
  if (cap_ok) {
    const int pages = (int)ceil_div64(L, kBlock);
    for (int p = tid; p < pages; p += blockDim.x) {
      const int id = bt[p];
      bad_block |= (id < 0 || id >= d.num_blocks);
    }
  }
  // topology
  int bad_topo = 0;
  if (parent != nullptr) {
    const int32_t* par = parent + (int64_t)b * d.M;
    for (int n = tid; n < d.M; n += blockDim.x) {
      const int pn = par[n];
      bad_topo |= (n == 0) ? (pn != -1) : (pn < 0 || pn >= n);
    }
  }
  bad_block = __syncthreads_or(bad_block);
  bad_topo = __syncthreads_or(bad_topo);
  const bool ok = cap_ok && !bad_block && !bad_topo;
  if (tid == 0) {
    req_ok[b] = ok ? 1 : 0;
    if (!cap_ok) raise_status(status, SPEC_ERR_CAPACITY);
    if (bad_block) raise_status(status, SPEC_ERR_DEVICE_BOUNDS);
    if (bad_topo) raise_status(status, SPEC_ERR_INVALID_ARG);
  }
  if (!ok) return;

  // append: positions ctx .. end-1 where end = ceil(L/16)*16; rows past
  // ctx+M-1 are cleared.
  constexpr int kVec = 16 / sizeof(T);
  const int lanes = d.D / kVec;  // 16-byte vectors per (position, head)
  const int64_t end = ceil_div64(L, kBlock) * kBlock;
  const int npos = (int)(end - ctx);
  const int work = npos * d.Hkv * lanes;
  for (int w = tid; w < work; w += blockDim.x) {
    const int lane = w % lanes;
    const int h = (w / lanes) % d.Hkv;
    const int i = w / (lanes * d.Hkv);
    const int64_t t = (int64_t)ctx + i;
    const int64_t dst = (((int64_t)bt[t / kBlock] * d.Hkv + h) * kBlock + t % kBlock) * d.D;
    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (i < d.M) {
      const int64_t src = (((int64_t)b * d.M + i) * d.Hkv + h) * d.D;
      kv = reinterpret_cast<const uint4*>(k_new + src)[lane];
      vv = reinterpret_cast<const uint4*>(v_new + src)[lane];
    }
    reinterpret_cast<uint4*>(k_cache + dst)[lane] = kv;
    reinterpret_cast<uint4*>(v_cache + dst)[lane] = vv;
  }
}

// ---------------------------------------------------------------------------
// split-KV attention on CUDA cores
// ---------------------------------------------------------------------------
// Shared-memory layout (floats):
//   qs [R][D]        queries pre-scaled by softmax_scale*log2(e)
//   ks [32][D+4]     key tile (row padding keeps 16-byte reads conflict-free)
//   vs [32][D]       value tile
//   ps [R][32]       probabilities of the tile
constexpr int kTileKeys = 32;
constexpr int kSimtThreads = 128;
constexpr int kSimtWarps = kSimtThreads / kWarp;
constexpr int kMaxRows = 128;  // new rows per request (tree nodes)

size_t attn_simt_smem_bytes(int R, int D) {
  return sizeof(float) * ((size_t)R * D + kTileKeys * (D + 4) + kTileKeys * D + (size_t)R * kTileKeys) +
         sizeof(unsigned long long) * 2 * kMaxRows;
}

template <typename T, int D, int RPW>
__global__ void __launch_bounds__(kSimtThreads) attn_split_kernel(
    const T* __restrict__ q, const T* __restrict__ k_cache, const T* __restrict__ v_cache,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ ctx_lens,
    const int32_t* __restrict__ parent, const int32_t* __restrict__ req_ok, spec_dims d,
    float qscale, int split_keys, int max_splits, float* __restrict__ part) {
  constexpr int DPL = D / kWarp;  // d values per lane in the PV step
  static_assert(DPL == 2 || DPL == 4, "D must be 64 or 128");
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (!req_ok[b]) return;
  const int ctx = ctx_lens[b];
  const int L = ctx + d.M;
  const int k0 = s * split_keys;
  if (k0 >= L) return;
  const int k1 = min(k0 + split_keys, L);
  const int group = d.Hq / d.Hkv;
  const int R = group * d.M;
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;

  extern __shared__ __align__(16) float smem[];
  float* qs = smem;
  float* ks = qs + R * D;
  float* vs = ks + kTileKeys * (D + 4);
  float* ps = vs + kTileKeys * D;
  // [row][2]: bits 0..63 and 64..127 of each row's mask
  unsigned long long* anc = reinterpret_cast<unsigned long long*>(ps + R * kTileKeys);

  // queries of the rows that read KV head h: row r = i*group + g
  for (int e = tid; e < R * D; e += kSimtThreads) {
    const int r = e / D, dd = e % D;
    const int i = r / group, hq = h * group + r % group;
    qs[e] = to_f32(q[(((int64_t)b * d.M + i) * d.Hq + hq) * D + dd]) * qscale;
  }
  // ancestor-or-self masks of the new rows
  for (int i = tid; i < d.M; i += kSimtThreads) {
    unsigned long long lo = 0, hi = 0;
    if (parent == nullptr) {
      lo = i >= 63 ? ~0ull : ((1ull << (i + 1)) - 1);
      hi = i >= 127 ? ~0ull : (i >= 64 ? ((1ull << (i - 63)) - 1) : 0ull);
    } else {
      // the append kernel has checked the topology (parent[n] < n), so
      // the walk reaches the root
      const int32_t* par = parent + (int64_t)b * d.M;
      for (int n = i, step = 0; step <= kMaxRows && n >= 0; ++step, n = par[n]) {
        if (n < 64) lo |= 1ull << n;
        else hi |= 1ull << (n - 64);
      }
    }
    anc[2 * i] = lo;
    anc[2 * i + 1] = hi;
  }

  float o[RPW][DPL];
  float mrow[RPW], lrow[RPW];
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    mrow[j] = -INFINITY;
    lrow[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[j][c] = 0.f;
  }

  const int32_t* bt = block_table + (int64_t)b * d.max_blocks;
  constexpr int kVec = 16 / sizeof(T);
  constexpr int kVecPerKey = D / kVec;

  for (int t0 = k0; t0 < k1; t0 += kTileKeys) {
    __syncthreads();  // previous tile fully consumed
    for (int e = tid; e < kTileKeys * kVecPerKey; e += kSimtThreads) {
      const int kk = e / kVecPerKey, vi = e % kVecPerKey;
      const int t = t0 + kk;
      float kf[kVec], vf[kVec];
      if (t < k1) {
        const int64_t base = (((int64_t)bt[t / kBlock] * d.Hkv + h) * kBlock + t % kBlock) * D;
        const uint4 kr = reinterpret_cast<const uint4*>(k_cache + base)[vi];
        const uint4 vr = reinterpret_cast<const uint4*>(v_cache + base)[vi];
        unpack16(kr, kf);
        unpack16(vr, vf);
      } else {
#pragma unroll
        for (int c = 0; c < kVec; ++c) kf[c] = vf[c] = 0.f;
      }
#pragma unroll
      for (int c = 0; c < kVec; ++c) {
        ks[kk * (D + 4) + vi * kVec + c] = kf[c];
        vs[kk * D + vi * kVec + c] = vf[c];
      }
    }
    __syncthreads();

    // scores: lane = key of the tile, rows warp + kSimtWarps*j
    const int t = t0 + lane;
    float sc[RPW];
#pragma unroll
    for (int j = 0; j < RPW; ++j) sc[j] = 0.f;
    const float4* krow = reinterpret_cast<const float4*>(ks + lane * (D + 4));
#pragma unroll 4
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 kv = krow[d4];
#pragma unroll
      for (int j = 0; j < RPW; ++j) {
        const int r = warp + kSimtWarps * j;
        if (r < R) {
          const float4 qv = reinterpret_cast<const float4*>(qs + r * D)[d4];
          sc[j] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      const int r = warp + kSimtWarps * j;
      if (r >= R) break;  // warp-uniform
      const int i = r / group;
      bool vis = t < k1;
      if (vis && t >= ctx) {
        const int k = t - ctx;  // new position, < M
        vis = (anc[2 * i + (k >> 6)] >> (k & 63)) & 1ull;
      }
      const float sj = vis ? sc[j] : -INFINITY;
      const float mnew = fmaxf(mrow[j], warp_max(sj));
      float p = 0.f, corr = 1.f;
      if (mnew != -INFINITY) {
        p = fast_exp2(sj - mnew);
        corr = exp2f(mrow[j] - mnew);
      }
      lrow[j] = lrow[j] * corr + warp_sum(p);
      mrow[j] = mnew;
      ps[r * kTileKeys + lane] = p;
#pragma unroll
      for (int c = 0; c < DPL; ++c) o[j][c] *= corr;
    }
    __syncwarp();
    // o[r][d] += sum_k p[r][k] * v[k][d], lane owns d = lane*DPL ..
#pragma unroll
    for (int k4 = 0; k4 < kTileKeys / 4; ++k4) {
      float4 p4[RPW];
#pragma unroll
      for (int j = 0; j < RPW; ++j) {
        const int r = warp + kSimtWarps * j;
        p4[j] = (r < R) ? reinterpret_cast<const float4*>(ps + r * kTileKeys)[k4]
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float vv[DPL];
        if constexpr (DPL == 4) {
          const float4 v4 = reinterpret_cast<const float4*>(vs + (k4 * 4 + kk) * D)[lane];
          vv[0] = v4.x; vv[1] = v4.y; vv[2] = v4.z; vv[3] = v4.w;
        } else {
          const float2 v2 = reinterpret_cast<const float2*>(vs + (k4 * 4 + kk) * D)[lane];
          vv[0] = v2.x; vv[1] = v2.y;
        }
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
          const float pk = kk == 0 ? p4[j].x : kk == 1 ? p4[j].y : kk == 2 ? p4[j].z : p4[j].w;
#pragma unroll
          for (int c = 0; c < DPL; ++c) o[j][c] += pk * vv[c];
        }
      }
    }
  }

  // partial: normalized O and log2-sum-exp per row
  float* pbase = part + (((int64_t)b * d.Hkv + h) * max_splits + s) * (int64_t)R * (D + 1);
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const int r = warp + kSimtWarps * j;
    if (r >= R) break;
    const float inv = lrow[j] > 0.f ? 1.f / lrow[j] : 0.f;
    float* prow = pbase + (int64_t)r * (D + 1);
#pragma unroll
    for (int c = 0; c < DPL; ++c) prow[lane * DPL + c] = o[j][c] * inv;
    if (lane == 0) prow[D] = lrow[j] > 0.f ? mrow[j] + log2f(lrow[j]) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// merge of the split partials
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) attn_combine_kernel(
    const float* __restrict__ part, const int32_t* __restrict__ ctx_lens,
    const int32_t* __restrict__ req_ok, spec_dims d, int split_keys, int max_splits,
    T* __restrict__ out, float* __restrict__ lse) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int group = d.Hq / d.Hkv;
  const int R = group * d.M;
  const int D = d.D;
  const bool ok = req_ok[b] != 0;
  const int L = ok ? ctx_lens[b] + d.M : 0;
  const int nsp = ok ? ceil_div(L, split_keys) : 0;
  const float* pbase = part + ((int64_t)b * d.Hkv + h) * max_splits * (int64_t)R * (D + 1);
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int nwarps = blockDim.x / kWarp;
  for (int r = warp; r < R; r += nwarps) {
    const int i = r / group, hq = h * group + r % group;
    float m = -INFINITY;
    for (int s = 0; s < nsp; ++s) m = fmaxf(m, pbase[((int64_t)s * R + r) * (D + 1) + D]);
    float wsum = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (m != -INFINITY) {
      for (int s = 0; s < nsp; ++s) {
        const float* prow = pbase + ((int64_t)s * R + r) * (D + 1);
        const float ls = prow[D];
        if (ls == -INFINITY) continue;
        const float w = exp2f(ls - m);
        wsum += w;
        for (int c = 0; c < D / kWarp; ++c) acc[c] += w * prow[lane + c * kWarp];
      }
    }
    T* orow = out + (((int64_t)b * d.M + i) * d.Hq + hq) * D;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    for (int c = 0; c < D / kWarp; ++c) orow[lane + c * kWarp] = from_f32<T>(acc[c] * inv);
    if (lse != nullptr && lane == 0) {
      lse[((int64_t)b * d.M + i) * d.Hq + hq] =
          wsum > 0.f ? (m + log2f(wsum)) * 0.69314718055994530942f : -INFINITY;
    }
  }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
cudaError_t kv_append_launch(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  const spec_dims& d = a.d;
  int32_t* req_ok = reinterpret_cast<int32_t*>(static_cast<char*>(a.ws) + lay.attn_ok_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<char*>(a.ws) + lay.status_off);
  PdlLaunch L(dim3(d.B), dim3(256), 0, st);
  cudaError_t e;
  if (d.kv_dtype == SPEC_BF16) {
    using T = __nv_bfloat16;
    e = cudaLaunchKernelEx(&L.cfg, kv_append_kernel<T>, static_cast<const T*>(a.k_new),
                           static_cast<const T*>(a.v_new), static_cast<T*>(a.k_cache),
                           static_cast<T*>(a.v_cache), a.block_table, a.ctx_lens, a.parent, d,
                           req_ok, status);
  } else {
    e = cudaLaunchKernelEx(&L.cfg, kv_append_kernel<float>, static_cast<const float*>(a.k_new),
                           static_cast<const float*>(a.v_new), static_cast<float*>(a.k_cache),
                           static_cast<float*>(a.v_cache), a.block_table, a.ctx_lens, a.parent,
                           d, req_ok, status);
  }
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
static cudaError_t launch_simt(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  const spec_dims& d = a.d;
  const int R = (d.Hq / d.Hkv) * d.M;
  int32_t* req_ok = reinterpret_cast<int32_t*>(static_cast<char*>(a.ws) + lay.attn_ok_off);
  float* part = reinterpret_cast<float*>(static_cast<char*>(a.ws) + lay.attn_off);

  kv_append_launch(a, lay, st, launches);

  const size_t smem = attn_simt_smem_bytes(R, d.D);
  const dim3 grid(lay.max_splits, d.Hkv, d.B);
  const float qscale = a.scale * 1.4426950408889634f;
  cudaError_t e = cudaSuccess;
#define SPECV_SIMT(DD, RPW)                                                                   \
  do {                                                                                        \
    auto k = attn_split_kernel<T, DD, RPW>;                                                   \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);      \
    if (e != cudaSuccess) return e;                                                           \
    k<<<grid, kSimtThreads, smem, st>>>(static_cast<const T*>(a.q),                           \
                                        static_cast<const T*>(a.k_cache),                     \
                                        static_cast<const T*>(a.v_cache), a.block_table,      \
                                        a.ctx_lens, a.parent, req_ok, d, qscale,              \
                                        lay.split_keys, lay.max_splits, part);                \
  } while (0)
  const int rpw = ceil_div(R, kSimtWarps);
  if (d.D == 128) {
    if (rpw <= 2) SPECV_SIMT(128, 2);
    else if (rpw <= 4) SPECV_SIMT(128, 4);
    else if (rpw <= 8) SPECV_SIMT(128, 8);
    else if (rpw <= 16) SPECV_SIMT(128, 16);
    else SPECV_SIMT(128, 32);
  } else {
    if (rpw <= 2) SPECV_SIMT(64, 2);
    else if (rpw <= 4) SPECV_SIMT(64, 4);
    else if (rpw <= 8) SPECV_SIMT(64, 8);
    else if (rpw <= 16) SPECV_SIMT(64, 16);
    else SPECV_SIMT(64, 32);
  }
#undef SPECV_SIMT
  ++*launches;

  attn_combine_kernel<T><<<dim3(d.Hkv, d.B), 256, 0, st>>>(
      part, a.ctx_lens, req_ok, d, lay.split_keys, lay.max_splits, static_cast<T*>(a.out), a.lse);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t attn_launch_simt(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  if (a.d.kv_dtype == SPEC_BF16) return launch_simt<__nv_bfloat16>(a, lay, st, launches);
  return launch_simt<float>(a, lay, st, launches);
}

}  // namespace specv
