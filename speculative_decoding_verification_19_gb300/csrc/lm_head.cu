// LM head with the reject-sample statistics in its epilogue.
//
// Page 2 §1.2: decoding is bound by the bytes it moves -- weights and the
// vocabulary-length logit rows.  The verify step's logits are the LM head
// z = h W^T of the M new rows of every request, for the target and for the
// draft model; the reject-sample statistics pass then reads every logit row
// once more.  Here the LM head itself forms those statistics (each row's
// maximum and scaled sum over every 2048-logit chunk, and the chunk's first
// argmax) from its fp32 accumulators while it writes the bf16 logits, so that
// the decisions start without a second pass over the rows.
//
// The GEMM (bf16 in, fp32 accumulate) runs on the tcgen05 tensor cores: one
// persistent CTA per SM, 8 warps:
//   warp 0      TMA producer: 128 x 64 tiles of h and 256 x 64 tiles of W
//               (128-byte swizzle) into a 4-stage ring of 48 KB;
//   warp 1      MMA issuer: D[128 x 256] += A B^T over the hidden size, four
//               K = 16 instructions per stage, into one of two TMEM
//               accumulators (2 x 256 columns);
//   warp 2      TMEM allocation;
//   warps 4-7   epilogue, one TMEM sub-partition (32 rows) each: the
//               accumulator read 32 columns at a time, rounded to bf16,
//               stored, and folded into the row's running chunk statistics.
// A unit is one 128-row tile by one 2048-column chunk (eight 256-column
// sub-tiles).  A CTA's work item is one of P equal pieces of a unit (P = 1,
// 2, 4 or 8, chosen at launch so that the items fill the last wave of CTAs):
// with P = 1 a chunk's statistics are complete inside one thread; with
// P > 1 every piece leaves its partial statistics in the workspace and the
// piece that finishes last (per 32-row warp, a fence and a counter) merges
// them in piece order.  Items are taken chunk-major with the row tile
// fastest, so the CTAs working at one time read the same W tiles (from L2
// after the first).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "lm_head.cuh"
#include "reject_sample.cuh"
#include "rs_device.cuh"
#include "tc_ptx.cuh"

namespace specv {
namespace lm {

constexpr int kBM = 128;               // rows of a tile (MMA M)
constexpr int kBN = 256;               // columns of a sub-tile (MMA N)
constexpr int kBK = 64;                // hidden elements per stage (one 128-byte row)
constexpr int kSubs = 8;               // sub-tiles per unit: 2048 columns
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kABytes = kBM * kBK * 2;                 // 16 KB
constexpr int kBBytes = kBN * kBK * 2;                 // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;         // 48 KB
constexpr int kTmemCols = 2 * kBN;                     // two accumulators
constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kAllocWarp = 2, kEpiWarp0 = 4;

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Work item w: piece p of unit (row tile mt, chunk nu), sub-tiles [j0, j1)
// of the row (empty for a piece past the end of a short last chunk).
struct Piece {
  int mt, nu, p, j0, j1;
  int64_t u;  // the unit, chunk-major
};

__device__ __forceinline__ Piece piece_of(int64_t w, int m_tiles, int P, int n_subs) {
  Piece q;
  q.mt = (int)(w % m_tiles);
  const int64_t rest = w / m_tiles;
  q.p = (int)(rest % P);
  q.nu = (int)(rest / P);
  q.u = (int64_t)q.nu * m_tiles + q.mt;
  const int per = kSubs / P;
  q.j0 = q.nu * kSubs + q.p * per;
  q.j1 = min(n_subs, q.j0 + per);
  if (q.j1 < q.j0) q.j1 = q.j0;
  return q;
}

// Row r of the logits / hidden states is node n = r % M of request r / M;
// its chunk statistics go where the reject-sample kernels read them (target
// rows: which = 0, draft rows: which = 1).
__global__ void __launch_bounds__(kThreads, 1) lm_head_kernel(
    const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int R,
    int H, int V, __nv_bfloat16* __restrict__ logits, RowStat* stats, int which, int M,
    int n_chunks, const float* temperature, spec_dims d, uint32_t* status, int P,
    RowStat* part, uint32_t* cnt) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ Bars bars_s;
  Bars* bars = &bars_s;
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const uint64_t wait = wait_limit_cycles(d);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[i]), 4);  // the four epilogue warps
    }
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_a);
    ptx::prefetch_tmap(&tm_b);
  }
  if (warp == kAllocWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  pdl_trigger();
  pdl_wait();  // the hidden states may come from the previous kernel

  const int m_tiles = (R + kBM - 1) / kBM;
  const int n_subs = V / kBN;                        // V is a multiple of 256
  const int n_units_n = (n_subs + kSubs - 1) / kSubs;
  const int64_t units = (int64_t)m_tiles * n_units_n;
  const int64_t items = units * P;
  const int kblocks = H / kBK;                       // H is a multiple of 64

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int64_t it = 0;
      bool ok = true;
      for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
        const Piece q = piece_of(w, m_tiles, P, n_subs);
        const int mt = q.mt;
        for (int j = q.j0; j < q.j1 && ok; ++j)
          for (int kb = 0; kb < kblocks; ++kb, ++it) {
            const int s = (int)(it % kStages);
            if (it >= kStages &&
                !ptx::mbar_wait(ptx::smem_u32(&bars->empty[s]),
                                (uint32_t)(((it / kStages) & 1) ^ 1), abort, wait)) {
              ok = false;
              break;
            }
            const uint32_t fb = ptx::smem_u32(&bars->full[s]);
            uint8_t* st = smem + (size_t)s * kStageBytes;
            ptx::mbar_arrive_expect_tx(fb, kStageBytes);
            tma_load_2d(ptx::smem_u32(st), &tm_a, fb, kb * kBK, mt * kBM);
            tma_load_2d(ptx::smem_u32(st + kABytes), &tm_b, fb, kb * kBK, j * kBN);
          }
      }
      // every copy issued lands before the CTA may exit
      for (int64_t v = it > kStages ? it - kStages : 0; v < it; ++v)
        ptx::mbar_drain(ptx::smem_u32(&bars->full[v % kStages]), (uint32_t)((v / kStages) & 1),
                        kDefaultWaitCycles);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      const uint64_t da0 = ptx::sdesc_sw128(ptx::smem_u32(smem), 16, 1024);
      const uint64_t db0 = ptx::sdesc_sw128(ptx::smem_u32(smem + kABytes), 16, 1024);
      int64_t it = 0, t = 0;
      bool ok = true;
      for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
        const Piece q = piece_of(w, m_tiles, P, n_subs);
        for (int j = q.j0; j < q.j1 && ok; ++j, ++t) {
          const int acc = (int)(t & 1);
          if (t >= 2 && !ptx::mbar_wait(ptx::smem_u32(&bars->acc_empty[acc]),
                                        (uint32_t)(((t >> 1) & 1) ^ 1), abort, wait)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t dcol = tmem + (uint32_t)(acc * kBN);
          for (int kb = 0; kb < kblocks; ++kb, ++it) {
            const int s = (int)(it % kStages);
            if (!ptx::mbar_wait(ptx::smem_u32(&bars->full[s]), (uint32_t)((it / kStages) & 1),
                                abort, wait)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t da = da0 + (uint64_t)((s * kStageBytes) >> 4);
            const uint64_t db = db0 + (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              ptx::mma_ss(dcol, da + (uint64_t)((kk * 32) >> 4), db + (uint64_t)((kk * 32) >> 4),
                          idesc, (kb | kk) != 0 ? 1u : 0u);
            ptx::mma_commit(ptx::smem_u32(&bars->empty[s]));
          }
          if (!ok) break;
          ptx::mma_commit(ptx::smem_u32(&bars->acc_full[acc]));
        }
      }
      // every MMA issued completes before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&bars->drain));
      ptx::mbar_drain(ptx::smem_u32(&bars->drain), 0, kDefaultWaitCycles);
    }
  } else if (warp >= kEpiWarp0) {
    const int sub = warp - kEpiWarp0;  // TMEM sub-partition: lanes 32 sub .. 32 sub + 31
    const uint32_t lane_base = tmem + ((uint32_t)(sub * 32) << 16);
    int64_t t = 0;
    for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
      const Piece q = piece_of(w, m_tiles, P, n_subs);
      const int nu = q.nu, mt = q.mt;
      const int row = mt * kBM + sub * 32 + lane;
      const bool valid = row < R;
      float cs = 1.f;
      bool greedy = false;
      if (stats != nullptr && valid) {
        const float temp = temperature[row / M];
        cs = stat_scale(temp);
        greedy = temp == 0.f;
      }
      float m_run = -INFINITY;
      dfloat s_run = df_make(0.f);
      int am_run = 0;  // column of the chunk's first maximum, inside the chunk
      bool ok = true;
      for (int j = q.j0; j < q.j1; ++j, ++t) {
        const int acc = (int)(t & 1);
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->acc_full[acc]),
                                                    (uint32_t)((t >> 1) & 1), abort, wait))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t col_base = lane_base + (uint32_t)(acc * kBN);
        __nv_bfloat16* out = logits + (int64_t)row * V + (int64_t)j * kBN;
        // pass 1: round to bf16, store, and the sub-tile's first maximum
        float mt_ = -INFINITY;
        int amt = 0;
#pragma unroll 1
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t r[32];
          ptx::tmem_ld32(col_base + cc * 32, r);
          ptx::tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float z = __uint_as_float((i & 1) ? (pk[i >> 1] & 0xffff0000u) : (pk[i >> 1] << 16));
            if (z > mt_) {
              mt_ = z;
              amt = cc * 32 + i;
            }
          }
          if (valid) {
            uint4* o = reinterpret_cast<uint4*>(out + cc * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              o[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        if (stats != nullptr) {
          // pass 2: the sum of exp2((z - m) cs) against the chunk's running
          // maximum (the accumulator read again; bf16-rounded values, as
          // the statistics pass would read them)
          const float m_new = fmaxf(m_run, mt_);
          if (m_run != -INFINITY && m_new > m_run)
            s_run = df_mul_f(s_run, fast_exp2((m_run - m_new) * cs));
          if (mt_ > m_run) am_run = (j - nu * kSubs) * kBN + amt;
          m_run = m_new;
          if (m_run != -INFINITY) {
#pragma unroll 1
            for (int cc = 0; cc < kBN / 32; ++cc) {
              uint32_t r[32];
              ptx::tmem_ld32(col_base + cc * 32, r);
              ptx::tmem_wait_ld();
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const uint32_t p = ptx::pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                s0 += fast_exp2((__uint_as_float(p << 16) - m_run) * cs);
                s1 += fast_exp2((__uint_as_float(p & 0xffff0000u) - m_run) * cs);
              }
              s_run = df_add(s_run, df_make(s0 + s1));
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->acc_empty[acc]));
      }
      if (!ok) break;
      if (stats == nullptr) continue;
      RowStat rs;
      rs.m = m_run;
      rs.pad = pack_index(am_run);
      rs.s = df_to_d(s_run);
      if (P > 1) {
        // this piece's partial statistics, then the count of the unit's
        // pieces finished (per warp: the warp's 32 rows); the last merges
        // the pieces in order -- the maximum, the first piece holding it
        // for the argmax, the sums rescaled to it
        RowStat* slot = part + ((((int64_t)which * units + q.u) * P) * kBM) + sub * 32 + lane;
        if (valid) slot[(int64_t)q.p * kBM] = rs;
        __threadfence();
        __syncwarp();
        uint32_t prev = 0;
        uint32_t* c = cnt + ((int64_t)which * units + q.u) * 4 + sub;
        if (lane == 0) prev = atomicAdd(c, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != (uint32_t)(P - 1)) continue;
        __threadfence();
        if (lane == 0) *c = 0u;  // ready for the next call
        if (!valid) continue;
        RowStat pc[kSubs];
#pragma unroll
        for (int k = 0; k < kSubs; ++k)
          if (k < P && k != q.p) pc[k] = ld_stat_cg(slot + (int64_t)k * kBM);
        float mm = -INFINITY;
#pragma unroll
        for (int k = 0; k < kSubs; ++k)
          if (k < P) mm = fmaxf(mm, k == q.p ? rs.m : pc[k].m);
        double sm = 0.0;
        float pad = pack_index(0);
        bool found = false;
#pragma unroll
        for (int k = 0; k < kSubs; ++k) {
          if (k >= P) continue;
          const RowStat x = k == q.p ? rs : pc[k];
          if (x.m != -INFINITY) sm += x.s * (double)fast_exp2((x.m - mm) * cs);
          if (!found && x.m == mm) {
            pad = x.pad;
            found = true;
          }
        }
        rs.m = mm;
        rs.pad = pad;
        rs.s = sm;
      }
      if (valid) {
        const int b = row / M, n = row - b * M;
        if (!greedy) rs.pad = pack_index(0);
        stats[(((int64_t)b * 2 + which) * M + n) * n_chunks + nu] = rs;
      }
    }
  }
  __syncthreads();
  if (tid == 0 && *abort) raise_status(status, SPEC_ERR_TIMEOUT);
  if (warp == kAllocWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace lm

static PFN_cuTensorMapEncodeTiled_v12000 lm_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A [rows, H] bf16 row-major matrix as 64 x box_rows tiles, 128-byte swizzle.
static bool lm_make_map(CUtensorMap* m, const void* base, int64_t rows, int H, int box_rows) {
  auto fn = lm_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {(cuuint32_t)lm::kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool lm_head_supported(int R, int H, int V) {
  return R >= 1 && H >= lm::kBK && H % lm::kBK == 0 && V >= lm::kBN && V % lm::kBN == 0;
}

// Pieces per unit: the P in {1, 2, 4, 8} (at most max_pieces) whose items
// take the fewest sub-tile rounds, ceil(units P / CTAs) * 8 / P; the smallest
// among equals (fewer merges).
static int lm_pieces(int64_t units, int sms, int max_pieces) {
  int best = 1;
  int64_t best_cost = -1;
  for (int P = 1; P <= max_pieces && P <= lm::kSubs; P *= 2) {
    const int64_t items = units * P;
    const int64_t ctas = items < sms ? items : sms;
    const int64_t cost = (items + ctas - 1) / ctas * (lm::kSubs / P);
    if (best_cost < 0 || cost < best_cost) {
      best = P;
      best_cost = cost;
    }
  }
  return best;
}

int64_t lm_head_units(int R, int V) {
  return (int64_t)((R + lm::kBM - 1) / lm::kBM) * ((V / lm::kBN + lm::kSubs - 1) / lm::kSubs);
}

cudaError_t lm_head_launch(const void* hidden, const void* weight, int R, int H, int V,
                           void* logits, RowStat* stats, int which, int M, int n_chunks,
                           const float* temperature, const spec_dims& d, uint32_t* status,
                           RowStat* part, uint32_t* cnt, cudaStream_t st, int* launches) {
  CUtensorMap ta, tb;
  if (!lm_make_map(&ta, hidden, R, H, lm::kBM) || !lm_make_map(&tb, weight, V, H, lm::kBN))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(lm::lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)lm::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t units = lm_head_units(R, V);
  // without statistics the pieces need no merge; with them, only as many
  // as the workspace holds partials for
  const int max_pieces = stats == nullptr ? lm::kSubs : (part != nullptr ? kLmMaxPieces : 1);
  const int P = lm_pieces(units, sms, max_pieces);
  const int64_t items = units * P;
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  PdlLaunch L(dim3(grid), dim3(lm::kThreads), lm::kSmem, st);
  e = cudaLaunchKernelEx(&L.cfg, lm::lm_head_kernel, ta, tb, R, H, V,
                         static_cast<__nv_bfloat16*>(logits), stats, which, M, n_chunks,
                         temperature, d, status, P, part, cnt);
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaGetLastError();
}

}  // namespace specv
