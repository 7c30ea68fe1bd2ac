// Device helpers shared by the reject-sample kernels: temperature check,
// vector loads of logits, the element weights of the sampling / residual
// laws, and the statistics of one chunk of a logits row.
#pragma once

#include <float.h>

#include "common.cuh"
#include "reject_sample.cuh"

namespace specv {

constexpr int kStatVecs = 8;  // 16-byte vectors per lane per statistics chunk

// ---------------------------------------------------------------------------
// Double-float arithmetic: a value hi + lo held as two fp32 numbers with
// |lo| <= ulp(hi) / 2, about 48 significant bits.  Built on the exact
// two-sum of Knuth (The Art of Computer Programming, vol. 2, 4.2.2) and the
// FMA-based two-product; used for long sums and scans instead of fp64,
// whose rate on this part is a small fraction of fp32's.  Every operation
// is rounded explicitly (__fadd_rn, __fmul_rn) so that no contraction or
// reassociation can break the error-free transformations.
// ---------------------------------------------------------------------------
struct dfloat {
  float hi, lo;
};
__device__ __forceinline__ dfloat df_make(float x) { return dfloat{x, 0.f}; }
__device__ __forceinline__ dfloat df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return dfloat{s, e};
}
__device__ __forceinline__ dfloat df_norm(float s, float e) {
  const float hi = __fadd_rn(s, e);
  return dfloat{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}
__device__ __forceinline__ dfloat df_add(dfloat x, dfloat y) {
  const dfloat s = df_two_sum(x.hi, y.hi);
  return df_norm(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ dfloat df_neg(dfloat x) { return dfloat{-x.hi, -x.lo}; }
__device__ __forceinline__ dfloat df_sub(dfloat x, dfloat y) { return df_add(x, df_neg(y)); }
__device__ __forceinline__ dfloat df_mul_f(dfloat x, float y) {
  const float p = __fmul_rn(x.hi, y);
  const float e = fmaf(x.lo, y, fmaf(x.hi, y, -p));
  return df_norm(p, e);
}
__device__ __forceinline__ bool df_gt(dfloat a, dfloat b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}
__device__ __forceinline__ float df_to_f(dfloat x) { return __fadd_rn(x.hi, x.lo); }
// a * b exactly, as a double-float (the rounding error by one FMA)
__device__ __forceinline__ dfloat df_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return dfloat{p, fmaf(a, b, -p)};
}
__device__ __forceinline__ double df_to_d(dfloat x) { return (double)x.hi + (double)x.lo; }
__device__ __forceinline__ dfloat df_shfl_xor(dfloat x, int o) {
  return dfloat{__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)};
}
__device__ __forceinline__ dfloat df_shfl(dfloat x, int src) {
  return dfloat{__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}
__device__ __forceinline__ dfloat df_warp_sum(dfloat x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = df_add(x, df_shfl_xor(x, o));
  return x;
}
// Inclusive warp scan in lane order.
__device__ __forceinline__ dfloat df_warp_scan(dfloat x) {
  const int lane = threadIdx.x % kWarp;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const dfloat y{__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
    if (lane >= o) x = df_add(x, y);
  }
  return x;
}

__device__ __forceinline__ bool temperature_ok(float T) {
  return T >= FLT_MIN && T <= FLT_MAX;  // normal, positive, finite (NaN fails)
}
// A request's temperature is valid when it is 0 (greedy: every row's law is
// the point mass on its largest logit, the smallest index among ties) or a
// positive normal finite value.
__device__ __forceinline__ bool temperature_valid(float T) { return T == 0.0f || temperature_ok(T); }
// log2(e) / T for the statistics; rows of a greedy request are still reduced
// (with a scale of 1) so that rows without a distribution are found.
__device__ __forceinline__ float stat_scale(float T) {
  return temperature_ok(T) ? 1.4426950408889634f / T : 1.0f;
}

// Index inside a chunk of the first element equal to the chunk's maximum m,
// the chunk held as chunk_stat holds it (lane l: vectors v * 32 + l).
// Comparisons are exact, so the smallest index among equal maxima wins.
template <typename T>
__device__ __forceinline__ int chunk_argmax(const uint4 (&raw)[kStatVecs], int nvalid, float m) {
  constexpr int EPV = 16 / sizeof(T);
  const int lane = threadIdx.x % kWarp;
  int best = 0x7fffffff;
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v) {
    float f[EPV];
    unpack16(raw[v], f);
#pragma unroll
    for (int i = 0; i < EPV; ++i) {
      const int e = (v * kWarp + lane) * EPV + i;
      if (e < nvalid && f[i] == m && e < best) best = e;
    }
  }
  return __reduce_min_sync(0xffffffffu, best);
}
// A chunk statistic written by an earlier kernel of the chain (or another
// SM), read through L2 by a load the compiler keeps after the dependency
// wait (volatile asm, memory clobber).
__device__ __forceinline__ RowStat ld_stat_cg(const RowStat* p) {
  unsigned long long lo, hi;
  asm volatile("ld.global.cg.v2.u64 {%0, %1}, [%2];" : "=l"(lo), "=l"(hi) : "l"(p) : "memory");
  RowStat r;
  r.m = __uint_as_float((uint32_t)lo);
  r.pad = __uint_as_float((uint32_t)(lo >> 32));
  r.s = __longlong_as_double((long long)hi);
  return r;
}

// The chunk statistics keep the argmax index in RowStat's spare word.
__device__ __forceinline__ float pack_index(int i) { return __int_as_float(i); }
__device__ __forceinline__ int unpack_index(float f) { return __float_as_int(f); }

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

// Whether element e (logit z) is in a filtered row's kept prefix (v, idx).
__device__ __forceinline__ bool kept_at(float z, int64_t e, float v, int idx) {
  return z > v || (z == v && e <= (int64_t)idx);
}
// No filter on either row of the law.
__device__ __forceinline__ void ctx_no_filter(DecideCtx& c) {
  c.vT = -INFINITY;
  c.vD = -INFINITY;
  c.iT = 0x7fffffff;
  c.iD = 0x7fffffff;
}

// Weight of element e of the node's sampling / residual law:
//   nrej == 0:  exp2((z - mT) * cs)                     (unnormalised p)
//   nrej >= 1:  max(0, P_{nrej-1} - q)                  (unnormalised residual)
// with P_0 = p and P_j = max(0, P_{j-1} - q) / Z_j; p and q are zero outside
// their rows' kept prefixes (filtered laws).
__device__ __forceinline__ float weight_of(float zt, float zd, int64_t e, const DecideCtx& c,
                                           int nrej) {
  float et = fast_exp2((zt - c.mT) * c.cs);
  if (!kept_at(zt, e, c.vT, c.iT)) et = 0.f;
  if (nrej == 0) return et;
  float qv = fast_exp2((zd - c.mD) * c.cs) * c.invSD;
  if (!kept_at(zd, e, c.vD, c.iD)) qv = 0.f;
  float P = et * c.invST;
  for (int j = 1; j < nrej; ++j) P = fmaxf(P - qv, 0.f) * c.invZ[j];
  return fmaxf(P - qv, 0.f);
}

// weight_of for laws without filters: the same operations in the same order
// (every token is kept), without the per-element index compares.
__device__ __forceinline__ float weight_plain(float zt, float zd, const DecideCtx& c, int nrej) {
  const float et = fast_exp2((zt - c.mT) * c.cs);
  if (nrej == 0) return et;
  const float qv = fast_exp2((zd - c.mD) * c.cs) * c.invSD;
  float P = et * c.invST;
  for (int j = 1; j < nrej; ++j) P = fmaxf(P - qv, 0.f) * c.invZ[j];
  return fmaxf(P - qv, 0.f);
}
// weight_of, or weight_plain when the law is known to have no filter.
template <bool kFilt>
__device__ __forceinline__ float weight_sel(float zt, float zd, int64_t e, const DecideCtx& c,
                                            int nrej) {
  return kFilt ? weight_of(zt, zd, e, c, nrej) : weight_plain(zt, zd, c, nrej);
}

// Mass of a chunk of the node's target row under exp2((z - mT) * cs), from
// its statistics.
__device__ __forceinline__ double chunk_mass(const RowStat& r, float mT, float cs) {
  return r.m == -INFINITY ? 0.0 : r.s * (double)fast_exp2((r.m - mT) * cs);
}

// Statistics of one chunk held by a warp: lane l holds the 16-byte vectors
// v * 32 + l (v < kStatVecs) of the chunk, of which the first `nvalid`
// elements are in the row.  Returns the chunk maximum m (every lane) and
// s = sum exp2((z - m) * cs) (every lane): fp32 partial sums per lane, then
// an fp32 tree over the lanes.  The lanes' sums of 64 terms in [0, 1]
// already bound the relative error near 1e-6 in the worst case (about 5e-7
// typically), which the tree's five levels do not change materially.
template <typename T>
__device__ __forceinline__ float chunk_stat(const uint4 (&raw)[kStatVecs], int nvalid, float cs,
                                            float* s_out) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kChunk = kWarp * kStatVecs * EPV;
  const int lane = threadIdx.x % kWarp;
  if (sizeof(T) == 2 && nvalid >= kChunk) {
    // full bf16 chunk: exact packed maximum, then four partial sums
    __nv_bfloat162 mx2 = *reinterpret_cast<const __nv_bfloat162*>(&raw[0].x);
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) {
      const uint32_t w4[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162*>(&w4[q]));
    }
    const float m = warp_max(fmaxf(__low2float(mx2), __high2float(mx2)));
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int v = 0; v < kStatVecs; ++v) {
        const uint32_t w4[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
        s0 += fast_exp2((__uint_as_float(w4[0] << 16) - m) * cs);
        s1 += fast_exp2((__uint_as_float(w4[0] & 0xffff0000u) - m) * cs);
        s2 += fast_exp2((__uint_as_float(w4[1] << 16) - m) * cs);
        s3 += fast_exp2((__uint_as_float(w4[1] & 0xffff0000u) - m) * cs);
        s0 += fast_exp2((__uint_as_float(w4[2] << 16) - m) * cs);
        s1 += fast_exp2((__uint_as_float(w4[2] & 0xffff0000u) - m) * cs);
        s2 += fast_exp2((__uint_as_float(w4[3] << 16) - m) * cs);
        s3 += fast_exp2((__uint_as_float(w4[3] & 0xffff0000u) - m) * cs);
      }
    }
    *s_out = warp_sum((s0 + s1) + (s2 + s3));
    return m;
  }
  float m = -INFINITY;
#pragma unroll
  for (int v = 0; v < kStatVecs; ++v) {
    if ((v * kWarp + lane) * EPV < nvalid) {
      float f[EPV];
      unpack16(raw[v], f);
#pragma unroll
      for (int i = 0; i < EPV; ++i) m = fmaxf(m, f[i]);
    }
  }
  m = warp_max(m);
  float sl = 0.f;
  if (m != -INFINITY) {
#pragma unroll
    for (int v = 0; v < kStatVecs; ++v) {
      if ((v * kWarp + lane) * EPV < nvalid) {
        float f[EPV];
        unpack16(raw[v], f);
#pragma unroll
        for (int i = 0; i < EPV; ++i) sl += fast_exp2((f[i] - m) * cs);  // z - m is exact
      }
    }
  }
  *s_out = warp_sum(sl);
  return m;
}

}  // namespace specv
