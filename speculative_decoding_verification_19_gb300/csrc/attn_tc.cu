// Verify attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// with TMA-staged paged K/V tiles.
//
// What is computed is the same as the CUDA-core kernels in attn.cu (page 1
// §2.1, page 2 §3.3, page 3 tree-attention section): every new row attends
// to the cached prefix and to its ancestors-or-self among the new rows.
//
// Shape of the work.  For one request b and KV head h, the R = group*M query
// rows that read h are stacked into one M=128 MMA tile (rows past R are zero
// padding), so every K/V byte is read from HBM once and used by all R rows:
// arithmetic intensity is R flop/byte, above what CUDA cores can serve at
// HBM speed for R >= ~16 and far below the tensor-core ridge.  The key axis
// of all (b, h) pairs is cut into 64-key tiles (4 blocks of 16), and the
// tiles of the whole batch are split evenly over one persistent CTA per SM;
// a pair that straddles two CTAs yields two partial results that a small
// kernel merges by log-sum-exp.
//
// Per CTA, warp-specialised:
//   warps 10 and 7 (8 when R > 64)  producers: Q of each pair by TMA;
//               the K and V pages of each tile into a 4-stage ring (32 KB per
//               stage) by 16-byte cp.async copies placed in the swizzled
//               operand layout
//   warp 11     MMA issuer of S = Q K^T into TMEM (four buffers)
//   warp 9      MMA issuer of O += P V, P read back from TMEM (aliasing S);
//               two issuing threads because each tcgen05.mma takes about 90
//               cycles to issue, and one thread issuing both products of a
//               tile was the kernel's bottleneck
//   warps 0..7  softmax: one thread per query row (TMEM lane) and per half
//               tile (32 keys); the two halves of a row swap their maxima
//               through shared memory, exp2, P written as bf16 into TMEM;
//               O is rescaled in TMEM only when the running maximum grows by
//               more than 2^8

// TMEM: S0..S3 cols [0,64) .. [192,256), O [256,384).  Four S buffers let
// Q K^T of tile t wait only for P V of tile t-4: the hand-off chain QK ->
// softmax -> PV -> QK of a buffer is spread over four tiles in flight (the
// K/V ring of four stages bounds the look-ahead to about three).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "attn.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace specv {
namespace tc {

constexpr int kTileKeys = 64;
constexpr int kPages = kTileKeys / kBlock;  // 4
constexpr int kStages = 4;
constexpr int kQBufs = 2;  // Q buffers (two: the next pair's Q loads while the current one runs)
constexpr int kThreads = 384;
// Warp roles.  A warp may only touch the TMEM lanes of its sub-partition
// (warp % 4).  Softmax warps 0..7: warp w serves rows 32*(w%4).. and the
// half w/4 of each tile's 64 keys.  The producer and the Q K^T issuer sit on
// sub-partitions 2 and 3, away from the softmax warps of rows 0..63 (the
// common case R <= 64); the P V issuer is warp 9; warp 7 (R <= 64) or 8
// copies K/V with the producer.
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 10;  // Q (TMA) and half of the K/V copies
// the other half of the K/V copies: warp 7 (sub-partition 3, away from the
// softmax warps) when rows 64..127 are padding, else warp 8
constexpr int kCopyWarpSmallR = 7;
constexpr int kCopyWarpLargeR = 8;
constexpr int kCopyThreads = 64;    // threads issuing K/V copies (warps 8 and 10)
constexpr int kMmaWarp = 11;  // issues Q K^T
constexpr int kPvWarp = 9;    // issues P V
constexpr int kBoxBytes = kBlock * 128;       // one page x 64 of D, bf16: 2 KB
constexpr int kHalfBytes = kPages * kBoxBytes;  // 8 KB
constexpr int kStageBytes = 4 * kHalfBytes;     // K lo, K hi, V lo, V hi
constexpr int kQHalfBytes = 128 * 128;          // 128 rows x 128 B
constexpr int kQBytes = 2 * kQHalfBytes;
constexpr int kSBufs = 4;  // S buffers in TMEM
constexpr int kTmemCols = 512;
constexpr int kOCol = kSBufs * kTileKeys;
constexpr uint64_t kTimeoutNs = 4000000000ull;  // SM clocks per wait (about 2 s)

struct __align__(8) Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full[kQBufs];
  uint64_t q_empty[kQBufs];
  uint64_t s_full[kSBufs];
  uint64_t p_full[kSBufs];
  uint64_t o_done[kSBufs];  // completion of PV(t) lands on o_done[t % kSBufs]
  uint64_t drain[2];  // the Q K^T issuer's and the P V issuer's last completion
  uint64_t xbar[4][2];       // per sub-partition, per tile parity: both halves' maxima
  float xmax[2][2][128];     // [tile parity][half][row]
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + kQBufs * kQBytes + sizeof(Bars) + 1024;

size_t smem_bytes() { return kSmemBytes; }

// Position in the flat tile sequence: request b, KV head h, tile of the pair.
struct Cursor {
  int b, h, tile, nt;
  __device__ void seek(int64_t g, const int32_t* ntiles, const int32_t* prefix, int B) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)prefix[mid] <= g) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    nt = ntiles[b];
    const int64_t off = g - prefix[b];
    h = (int)(off / nt);
    tile = (int)(off % nt);
  }
  __device__ void next(const int32_t* ntiles, int B, int Hkv) {
    if (++tile < nt) return;
    tile = 0;
    if (++h < Hkv) return;
    h = 0;
    do {
      ++b;
    } while (b < B && ntiles[b] == 0);
    nt = b < B ? ntiles[b] : 0;
  }
};

// Scaled score of tile column j (log2 units) or -inf where the key is not
// visible to this row: past the tile's valid keys or the request's length,
// or a new position that is not an ancestor-or-self of the row's node.
__device__ __forceinline__ float score_of(uint32_t sbits, int j, int kpos0, int nkeys, int ctx,
                                          int L, unsigned long long anc, bool real, bool plain,
                                          float qscale2) {
  const float x = __uint_as_float(sbits) * qscale2;
  if (plain) return real ? x : -INFINITY;
  const int pos = kpos0 + j;
  bool vis = real && j < nkeys && pos < L;
  if (vis && pos >= ctx) vis = (anc >> (pos - ctx)) & 1ull;
  return vis ? x : -INFINITY;
}

__device__ __forceinline__ int tile_pages(int L, int tile) {
  const int keys = L - tile * kTileKeys;
  return keys >= kTileKeys ? kPages : ceil_div(keys, kBlock);
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __nv_bfloat16* __restrict__ k_cache,
    const __nv_bfloat16* __restrict__ v_cache, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ ctx_lens, const int32_t* __restrict__ parent,
    const int32_t* __restrict__ ntiles, const int32_t* __restrict__ prefix, spec_dims d,
    float qscale2, float* __restrict__ part, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* qbufs = smem + kStages * kStageBytes;
  Bars* bars = reinterpret_cast<Bars*>(qbufs + kQBufs * kQBytes);

  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  const int B = d.B, Hkv = d.Hkv, M = d.M;
  const int group = d.Hq / d.Hkv;
  const int R = group * M;
  const int G = gridDim.x, c = blockIdx.x;
  const int n_sm_warps = ceil_div(R, 32);
  pdl_trigger();

  // Set-up that needs nothing from the previous kernels runs while they
  // drain: Q padding, barriers, TMEM, tensor-map prefetch.
  // zero the Q buffers once: rows R..127 stay zero padding
  for (int i = tid; i < kQBufs * kQBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(qbufs)[i] = make_uint4(0, 0, 0, 0);
  ptx::fence_proxy_async_smem();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[s]), kCopyThreads);
      ptx::mbar_init(ptx::smem_u32(&bars->empty[s]), 1);
    }
    for (int i = 0; i < kQBufs; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->q_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->q_empty[i]), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->p_full[i]), 2 * n_sm_warps);
      ptx::mbar_init(ptx::smem_u32(&bars->o_done[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->drain[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain[1]), 1);
    for (int sp = 0; sp < 4; ++sp)
      for (int i = 0; i < 2; ++i) ptx::mbar_init(ptx::smem_u32(&bars->xbar[sp][i]), 2);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;

  pdl_wait();  // the tile plan and the appended rows come from the previous kernels
  const int64_t T = prefix[B];
  const int64_t g0 = (int64_t)c * T / G, g1 = (int64_t)(c + 1) * T / G;
  if (g0 >= g1) {  // uniform: no tiles for this CTA
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
    return;
  }

  const int copy_warp = n_sm_warps <= 2 ? kCopyWarpSmallR : kCopyWarpLargeR;
  if (warp == kProducerWarp || warp == copy_warp) {
    // ------------------------------------------------------------ producers
    // Both warps walk the tiles; lane j holds the four block ids of tile
    // (window start + j), fetched for 32 tiles at once.  Q comes by TMA
    // (warp 10, lane 0).  K and V come by 16-byte cp.async copies from all
    // 64 threads, each placed where the 128-byte-swizzled layout of the MMA
    // operands wants it (chunk j of row r of a page at j ^ (r % 8)): one
    // tensor-TMA box per page half and tensor bounded the kernel at about
    // 16 boxes per tile, whatever their size.
    const int ct = (warp == copy_warp ? 0 : kWarp) + lane;  // copy thread 0..63
    const int c16 = ct & 15;                                 // 16-byte chunk of a 256-byte row
    const int r0 = ct >> 4;                                  // rows r0, r0 + 4, r0 + 8, r0 + 12
    const uint32_t swz_half = (uint32_t)(c16 >> 3) * kHalfBytes;
    Cursor cu;
    cu.seek(g0, ntiles, prefix, B);
    int seg = -1, L = 0, win = -1;
    int ids[kPages] = {0, 0, 0, 0};
    int64_t t = 0;
    bool ok = true;
    for (int64_t g = g0; g < g1 && ok; ++g, ++t) {
      const bool first = (g == g0) || cu.tile == 0;
      if (first) {
        ++seg;
        L = ctx_lens[cu.b] + M;
        win = -1;
        if (warp == kProducerWarp) {
          if (lane == 0) {
            const int qb = seg % kQBufs;
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_empty[qb]), ((seg / kQBufs) & 1) ^ 1, abort,
                                kTimeoutNs);
            if (ok) {
              const uint32_t qf = ptx::smem_u32(&bars->q_full[qb]);
              ptx::mbar_arrive_expect_tx(qf, 2u * R * 128u);
              for (int half = 0; half < 2; ++half)
                ptx::tma_load_4d(ptx::smem_u32(qbufs + qb * kQBytes + half * kQHalfBytes), &tm_q,
                                 qf, half * 64, cu.h * group, 0, cu.b);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
      }
      if ((cu.tile >> 5) != win) {  // next window of 32 tiles of this pair
        win = cu.tile >> 5;
        const int page0 = ((win << 5) + lane) * kPages;
        const int32_t* bt = block_table + (int64_t)cu.b * d.max_blocks;
#pragma unroll
        for (int p = 0; p < kPages; ++p)
          ids[p] = (page0 + p < d.max_blocks) ? bt[page0 + p] : 0;
      }
      const int np = tile_pages(L, cu.tile);
      const int src = cu.tile & 31;
      int blk[kPages];
#pragma unroll
      for (int p = 0; p < kPages; ++p) blk[p] = __shfl_sync(0xffffffffu, ids[p], src);
      const int stage = (int)(t % kStages);
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty[stage]), (uint32_t)((t / kStages) & 1) ^ 1u,
                          abort, kTimeoutNs);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint32_t sb = ptx::smem_u32(stages + stage * kStageBytes);
#pragma unroll
      for (int p = 0; p < kPages; ++p) {
        if (p < np) {
          const int64_t page = ((int64_t)blk[p] * Hkv + cu.h) * kBlock;  // row of slot 0
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = r0 + 4 * k;
            const int64_t e = (page + r) * 128 + c16 * 8;  // element offset in the cache
            const uint32_t so = swz_half + (uint32_t)p * kBoxBytes + (uint32_t)r * 128u +
                                ((uint32_t)((c16 & 7) ^ (r & 7)) << 4);
            ptx::cp_async16(sb + so, k_cache + e);
            ptx::cp_async16(sb + 2 * kHalfBytes + so, v_cache + e);
          }
        }
      }
      ptx::cp_async_arrive_noinc(ptx::smem_u32(&bars->full[stage]));
      cu.next(ntiles, B, Hkv);
    }
    if (warp == kProducerWarp && lane == 0) {
      // every load issued must have landed before the CTA may exit
      const int64_t issued = t;  // a broken loop did not issue tile t
      for (int64_t u = issued > kStages ? issued - kStages : 0; u < issued; ++u)
        ptx::mbar_wait(ptx::smem_u32(&bars->full[u % kStages]), (uint32_t)((u / kStages) & 1),
                       abort, kTimeoutNs);
      for (int sg = seg >= kQBufs ? seg - kQBufs + 1 : 0; sg <= seg; ++sg)
        ptx::mbar_wait(ptx::smem_u32(&bars->q_full[sg % kQBufs]), (uint32_t)((sg / kQBufs) & 1),
                       abort, kTimeoutNs);
    }
    // the copies of a thread that stopped early land before the CTA exits
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA: Q K^T
    if (lane == 0) {
      const uint32_t id_qk_full = ptx::idesc_bf16_f32(128, kTileKeys, false, false);
      Cursor cu;
      cu.seek(g0, ntiles, prefix, B);
      int seg = -1, L = 0;
      int64_t t = 0;
      // Shared-memory descriptors built once; an operand at byte offset o
      // from a base is the base descriptor plus o >> 4 in the start-address
      // field (shared addresses stay below 2^18, so the 14-bit field never
      // carries).
      const uint64_t dq0 = ptx::sdesc_sw128(ptx::smem_u32(qbufs), 16, 1024);
      const uint64_t dk0 = ptx::sdesc_sw128(ptx::smem_u32(stages), 16, 1024);
      for (int64_t g = g0; g < g1; ++g, ++t) {
        const bool first = (g == g0) || cu.tile == 0;
        const bool last = (g == g1 - 1) || cu.tile == cu.nt - 1;
        if (first) ++seg;
        const int qb = seg % kQBufs;
        if (first && !ptx::mbar_wait(ptx::smem_u32(&bars->q_full[qb]),
                                     (uint32_t)((seg / kQBufs) & 1), abort, kTimeoutNs))
          break;
        const int stage = (int)(t % kStages);
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->full[stage]), (uint32_t)((t / kStages) & 1),
                            abort, kTimeoutNs))
          break;
        // PV(t - kSBufs) read P out of the S buffer this tile's QK writes
        if (t >= kSBufs && !ptx::mbar_wait(ptx::smem_u32(&bars->o_done[t % kSBufs]),
                                           (uint32_t)(((t - kSBufs) / kSBufs) & 1), abort,
                                           kTimeoutNs))
          break;
        ptx::tc_fence_after();
        if (first) L = ctx_lens[cu.b] + M;
        const int np = tile_pages(L, cu.tile);
        const uint32_t idqk = np == kPages ? id_qk_full : ptx::idesc_bf16_f32(128, np * 16, false, false);
        const uint64_t dq = dq0 + (uint64_t)((qb * kQBytes) >> 4);
        const uint64_t dk = dk0 + (uint64_t)((stage * kStageBytes) >> 4);
        const int sbuf = (int)(t % kSBufs);
        const uint32_t scol = tmem + sbuf * kTileKeys;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = dq + (uint64_t)(((k >> 2) * kQHalfBytes + (k & 3) * 32) >> 4);
          const uint64_t bd = dk + (uint64_t)(((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4);
          ptx::mma_ss(scol, ad, bd, idqk, k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->s_full[sbuf]));
        if (last) ptx::mma_commit(ptx::smem_u32(&bars->q_empty[qb]));
        cu.next(ntiles, B, Hkv);
      }
      // all MMAs issued by this thread complete before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&bars->drain[0]));
      ptx::mbar_wait(ptx::smem_u32(&bars->drain[0]), 0, abort, kTimeoutNs);
    }
  } else if (warp == kPvWarp) {
    // ---------------------------------------------------------------- MMA: P V
    // A second issuing thread, so that the two products of a tile are issued
    // side by side.  PV(u) follows the softmax of tile u (p_full) and frees the
    // tile's stage and its S buffer when it completes.
    if (lane == 0) {
      const uint32_t id_pv = ptx::idesc_bf16_f32(128, 128, false, true);
      const uint64_t dv0 = ptx::sdesc_sw128(ptx::smem_u32(stages + 2 * kHalfBytes), kHalfBytes, 1024);
      Cursor cu;
      cu.seek(g0, ntiles, prefix, B);
      int L = 0;
      int64_t u = 0;
      for (int64_t g = g0; g < g1; ++g, ++u) {
        const bool first = (g == g0) || cu.tile == 0;
        if (first) L = ctx_lens[cu.b] + M;
        const int np = tile_pages(L, cu.tile);
        const int sbuf = (int)(u % kSBufs);
        const int stage = (int)(u % kStages);
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->p_full[sbuf]), (uint32_t)((u / kSBufs) & 1), abort,
                            kTimeoutNs))
          break;
        ptx::tc_fence_after();
        const uint64_t dv = dv0 + (uint64_t)((stage * kStageBytes) >> 4);
        const uint32_t pcol = tmem + sbuf * kTileKeys;
#pragma unroll
        for (int j = 0; j < kPages; ++j) {
          if (j < np)
            ptx::mma_ts(tmem + kOCol, pcol + j * 8, dv + (uint64_t)((j * 2 * 1024) >> 4), id_pv,
                        (first && j == 0) ? 0u : 1u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->o_done[sbuf]));
        ptx::mma_commit(ptx::smem_u32(&bars->empty[stage]));
        cu.next(ntiles, B, Hkv);
      }
      ptx::mma_commit(ptx::smem_u32(&bars->drain[1]));
      ptx::mbar_wait(ptx::smem_u32(&bars->drain[1]), 0, abort, kTimeoutNs);
    }
  } else if (warp < kSoftmaxWarps) {
    // -------------------------------------------------------------- softmax
    const int sp = warp & 3;   // TMEM sub-partition this warp may access
    const int half = warp >> 2;  // keys [32*half, 32*half + 32) of each tile
    const int row = sp * 32 + lane;
    if (sp < n_sm_warps) {
      const uint32_t lane_base = tmem + ((uint32_t)(sp * 32) << 16);
      Cursor cu;
      cu.seek(g0, ntiles, prefix, B);
      int64_t t = 0;
      float m_used = -INFINITY, l = 0.f;
      unsigned long long anc = 0;
      int ctx = 0, L = 0;
      const bool real = row < R;
      for (int64_t g = g0; g < g1; ++g, ++t) {
        const bool first = (g == g0) || cu.tile == 0;
        const bool last = (g == g1 - 1) || cu.tile == cu.nt - 1;
        if (first) {
          ctx = ctx_lens[cu.b];
          L = ctx + M;
          m_used = -INFINITY;
          l = 0.f;
          anc = 0;
          if (real) {
            const int i = row / group;
            if (parent == nullptr) {
              anc = (i >= 63) ? ~0ull : ((1ull << (i + 1)) - 1);
            } else {
              const int32_t* par = parent + (int64_t)cu.b * M;
              int n = i;
              for (int step = 0; step <= 64 && n >= 0; ++step) {
                anc |= 1ull << n;
                n = par[n];
              }
            }
          }
        }
        const int sbuf = (int)(t % kSBufs);  // S / P buffer in TMEM
        const int xb = (int)(t & 1);          // maxima exchange buffer
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->s_full[sbuf]), (uint32_t)((t / kSBufs) & 1), abort,
                            kTimeoutNs))
          break;
        ptx::tc_fence_after();
        const int kpos0 = cu.tile * kTileKeys;
        const int nkeys = tile_pages(L, cu.tile) * kBlock;
        // tiles wholly inside the cached prefix need no mask
        const bool plain = kpos0 + kTileKeys <= ctx && nkeys == kTileKeys;
        const int jbase = half * 32;
        uint32_t sv[32];
        ptx::tmem_ld32(lane_base + sbuf * kTileKeys + jbase, sv);
        ptx::tmem_wait_ld();
        // maximum of this half (log2 units), then of the whole tile
        float mh;
        if (plain) {
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            a0 = fmaxf(a0, __uint_as_float(sv[j]));
            a1 = fmaxf(a1, __uint_as_float(sv[j + 1]));
            a2 = fmaxf(a2, __uint_as_float(sv[j + 2]));
            a3 = fmaxf(a3, __uint_as_float(sv[j + 3]));
          }
          mh = real ? fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * qscale2 : -INFINITY;
        } else {
          mh = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            mh = fmaxf(mh, score_of(sv[j], jbase + j, kpos0, nkeys, ctx, L, anc, real, false, qscale2));
        }
        bars->xmax[xb][half][row] = mh;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->xbar[sp][xb]));
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->xbar[sp][xb]), (uint32_t)((t >> 1) & 1), abort,
                            kTimeoutNs))
          break;
        const float mt = fmaxf(bars->xmax[xb][0][row], bars->xmax[xb][1][row]);
        bool need = false;
        if (first) {
          m_used = mt;
        } else if (mt > m_used + 8.0f) {
          need = true;
        }
        if (__any_sync(0xffffffffu, need)) {
          // O is rescaled in place (this half's 64 columns): PV(t-1) must have landed
          if (!ptx::mbar_wait(ptx::smem_u32(&bars->o_done[(t - 1) % kSBufs]),
                              (uint32_t)(((t - 1) / kSBufs) & 1), abort, kTimeoutNs))
            break;
          ptx::tc_fence_after();
          const float f = need ? exp2f(m_used - mt) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            const uint32_t oc = lane_base + kOCol + half * 64 + cc * 32;
            ptx::tmem_ld32(oc, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            ptx::tmem_st32(oc, o);
          }
          ptx::tmem_wait_st();
          if (need) {
            l *= f;
            m_used = mt;
          }
        }
        // probabilities of this half, packed to bf16 pairs; keys
        // 32*half.. land in P columns 16*half.. (S columns both halves have
        // already read, by the exchange above)
        uint32_t pk[16];
        float l0 = 0.f, l1 = 0.f;
        if (plain) {
          const float nm = real ? -m_used : -INFINITY;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float pa = fast_exp2(fmaf(__uint_as_float(sv[2 * j]), qscale2, nm));
            const float pb = fast_exp2(fmaf(__uint_as_float(sv[2 * j + 1]), qscale2, nm));
            l0 += pa;
            l1 += pb;
            pk[j] = ptx::pack_bf16x2(pa, pb);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float xa = score_of(sv[2 * j], jbase + 2 * j, kpos0, nkeys, ctx, L, anc, real,
                                      false, qscale2);
            const float xb = score_of(sv[2 * j + 1], jbase + 2 * j + 1, kpos0, nkeys, ctx, L, anc,
                                      real, false, qscale2);
            const float pa = xa == -INFINITY ? 0.f : fast_exp2(xa - m_used);
            const float pb = xb == -INFINITY ? 0.f : fast_exp2(xb - m_used);
            l0 += pa;
            l1 += pb;
            pk[j] = ptx::pack_bf16x2(pa, pb);
          }
        }
        l += l0 + l1;
        ptx::tmem_st16(lane_base + sbuf * kTileKeys + half * 16, pk);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full[sbuf]));
        if (last) {
          if (!ptx::mbar_wait(ptx::smem_u32(&bars->o_done[sbuf]), (uint32_t)((t / kSBufs) & 1),
                              abort, kTimeoutNs))
            break;
          ptx::tc_fence_after();
          // partial: unnormalised O (this half's 64 columns), the running
          // maximum and this half's share of the row sum
          const int64_t slot = (int64_t)cu.b * Hkv + cu.h + c;
          float* prow = part + (slot * R + (real ? row : 0)) * (int64_t)tc_part_stride(d.D);
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            ptx::tmem_ld32(lane_base + kOCol + half * 64 + cc * 32, o);
            ptx::tmem_wait_ld();
            if (real) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                const float4 v = make_float4(__uint_as_float(o[j]), __uint_as_float(o[j + 1]),
                                             __uint_as_float(o[j + 2]), __uint_as_float(o[j + 3]));
                *reinterpret_cast<float4*>(prow + half * 64 + cc * 32 + j) = v;
              }
            }
          }
          if (real) {
            prow[d.D + 1 + half] = l;
            if (half == 0) prow[d.D] = m_used;
          }
          ptx::tc_fence_before();
        }
        cu.next(ntiles, B, Hkv);
      }
    }
  }

  __syncthreads();
  if (tid == 0 && *abort) raise_status(status, SPEC_ERR_TIMEOUT);
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// plan: tiles per request and their exclusive prefix over (request, head)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) attn_plan_kernel(const int32_t* __restrict__ ctx_lens,
                                                         const int32_t* __restrict__ req_ok,
                                                         spec_dims d, int32_t* __restrict__ ntiles,
                                                         int32_t* __restrict__ prefix) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  pdl_trigger();
  pdl_wait();  // the append's per-request verdicts
  const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < d.B; base += 1024) {
    const int b = base + tid;
    int nt = 0;
    if (b < d.B && req_ok[b]) nt = ceil_div(ctx_lens[b] + d.M, kTileKeys);
    if (b < d.B) ntiles[b] = nt;
    int v = nt * d.Hkv;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int wpre = 0;
    for (int i = 0; i < warp; ++i) wpre += warp_tot[i];
    const int c0 = carry;
    if (b < d.B) prefix[b] = c0 + wpre + incl - v;
    __syncthreads();
    if (tid == 1023) carry = c0 + wpre + incl;
    __syncthreads();
  }
  if (tid == 0) prefix[d.B] = carry;
}

// ---------------------------------------------------------------------------
// merge of the partials of each (request, KV head)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) attn_tc_combine_kernel(
    const float* __restrict__ part, const int32_t* __restrict__ ntiles,
    const int32_t* __restrict__ prefix, spec_dims d, int G, T* __restrict__ out,
    float* __restrict__ lse) {
  // one warp per query row: blockIdx.x = group of 4 rows, y = KV head, z = request
  const int h = blockIdx.y, b = blockIdx.z;
  const int group = d.Hq / d.Hkv;
  const int R = group * d.M;
  const int D = d.D;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int r = blockIdx.x * (blockDim.x / kWarp) + warp;
  pdl_trigger();
  pdl_wait();  // the partials come from the previous kernel
  if (r >= R) return;
  const int64_t Ttot = prefix[d.B];
  const int nt = ntiles[b];
  int c_first = 1, c_last = 0;
  if (nt > 0) {
    const int64_t ps = (int64_t)prefix[b] + (int64_t)h * nt, pe = ps + nt;
    c_first = (int)(((ps + 1) * G - 1) / Ttot);
    c_last = (int)((pe * G - 1) / Ttot);
  }
  const int64_t pair = (int64_t)b * d.Hkv + h;
  const int i = r / group, hq = h * group + r % group;
  // A partial row holds unnormalised O, the running maximum m (log2 units)
  // and the two half-tile shares of the row sum.  CTAs with an empty tile
  // range wrote nothing (their slot may belong to a neighbouring pair), so
  // they are skipped.  Lane c reads the scalars of partial c_first + c (all
  // partials in one round trip), then every lane its D / 32 values of each.
  const int S = tc_part_stride(D);
  const int np = c_last - c_first + 1;
  float m = -INFINITY;
  for (int c0 = 0; c0 < np; c0 += kWarp) {
    const int cc = c_first + c0 + lane;
    float mc = -INFINITY;
    if (c0 + lane < np && (int64_t)cc * Ttot / G != (int64_t)(cc + 1) * Ttot / G) {
      const float* prow = part + ((pair + cc) * R + r) * (int64_t)S;
      if (prow[D + 1] + prow[D + 2] > 0.f) mc = prow[D];
    }
    m = fmaxf(m, warp_max(mc));
  }
  float wsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (m != -INFINITY) {
    for (int cc = c_first; cc <= c_last; ++cc) {
      if ((int64_t)cc * Ttot / G == (int64_t)(cc + 1) * Ttot / G) continue;
      const float* prow = part + ((pair + cc) * R + r) * (int64_t)S;
      const float lp = prow[D + 1] + prow[D + 2];
      if (!(lp > 0.f)) continue;
      const float w = exp2f(prow[D] - m);
      wsum += w * lp;
      for (int k = 0; k < D / kWarp; ++k) acc[k] += w * prow[lane + k * kWarp];
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  T* orow = out + (((int64_t)b * d.M + i) * d.Hq + hq) * D;
  for (int k = 0; k < D / kWarp; ++k) orow[lane + k * kWarp] = from_f32<T>(acc[k] * inv);
  if (lse != nullptr && lane == 0)
    lse[((int64_t)b * d.M + i) * d.Hq + hq] =
        wsum > 0.f ? (m + log2f(wsum)) * 0.69314718055994530942f : -INFINITY;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

static bool make_map(CUtensorMap* m, const void* base, const cuuint64_t dims[4],
                     const cuuint64_t strides[3], const cuuint32_t box[4]) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

size_t attn_tc_part_floats(const spec_dims& d) {
  const int R = (d.Hq / d.Hkv) * d.M;
  return ((size_t)d.B * d.Hkv + kMaxAttnCtas) * R * tc_part_stride(d.D);
}

cudaError_t attn_launch_tc(const AttnArgs& a, const WsLayout& lay, cudaStream_t st, int* launches) {
  using namespace tc;
  const spec_dims& d = a.d;
  const int group = d.Hq / d.Hkv;
  char* ws = static_cast<char*>(a.ws);
  int32_t* req_ok = reinterpret_cast<int32_t*>(ws + lay.attn_ok_off);
  int32_t* ntiles = reinterpret_cast<int32_t*>(ws + lay.tc_ntiles_off);
  int32_t* prefix = reinterpret_cast<int32_t*>(ws + lay.tc_prefix_off);
  float* part = reinterpret_cast<float*>(ws + lay.attn_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + lay.status_off);

  CUtensorMap tm_q, tm_k, tm_v;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)d.D, (cuuint64_t)d.Hq, (cuuint64_t)d.M, (cuuint64_t)d.B};
    const cuuint64_t strides[3] = {(cuuint64_t)d.D * 2, (cuuint64_t)d.Hq * d.D * 2,
                                   (cuuint64_t)d.M * d.Hq * d.D * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)group, (cuuint32_t)d.M, 1};
    if (!make_map(&tm_q, a.q, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)d.D, (cuuint64_t)kBlock, (cuuint64_t)d.Hkv,
                                (cuuint64_t)d.num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)d.D * 2, (cuuint64_t)kBlock * d.D * 2,
                                   (cuuint64_t)d.Hkv * kBlock * d.D * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)kBlock, 1, 1};
    if (!make_map(&tm_k, a.k_cache, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map(&tm_v, a.v_cache, dims, strides, box)) return cudaErrorInvalidValue;
  }

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int G = sms < kMaxAttnCtas ? sms : kMaxAttnCtas;

  kv_append_launch(a, lay, st, launches);
  {
    PdlLaunch L(dim3(1), dim3(1024), 0, st);
    e = cudaLaunchKernelEx(&L.cfg, attn_plan_kernel, a.ctx_lens, (const int32_t*)req_ok, d, ntiles,
                           prefix);
    if (e != cudaSuccess) return e;
  }
  ++*launches;
  e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const float qscale2 = a.scale * 1.4426950408889634f;
  {
    PdlLaunch L(dim3(G), dim3(kThreads), kSmemBytes, st);
    e = cudaLaunchKernelEx(&L.cfg, attn_tc_kernel, tm_q, tm_k, tm_v,
                           static_cast<const __nv_bfloat16*>(a.k_cache),
                           static_cast<const __nv_bfloat16*>(a.v_cache), a.block_table, a.ctx_lens,
                           a.parent, (const int32_t*)ntiles, (const int32_t*)prefix, d, qscale2,
                           part, status);
    if (e != cudaSuccess) return e;
  }
  ++*launches;
  {
    const int R = (d.Hq / d.Hkv) * d.M;
    PdlLaunch L(dim3((R + 3) / 4, d.Hkv, d.B), dim3(128), 0, st);
    e = cudaLaunchKernelEx(&L.cfg, attn_tc_combine_kernel<__nv_bfloat16>, (const float*)part,
                           (const int32_t*)ntiles, (const int32_t*)prefix, d, G,
                           static_cast<__nv_bfloat16*>(a.out), a.lse);
    if (e != cudaSuccess) return e;
  }
  ++*launches;
  return cudaGetLastError();
}

}  // namespace specv
