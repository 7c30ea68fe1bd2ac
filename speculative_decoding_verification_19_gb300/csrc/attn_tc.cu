// Verify attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// with cp.async-staged paged K/V tiles.
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
// tiles of the whole batch are split over one persistent CTA per SM.
//
// Two launches per call:
//   attn_prep_kernel  one CTA per request: checks it (capacity, block ids,
//                     topology) and, for a tree, the ancestor-or-self mask
//                     of every row.  The last CTA
//                     to finish plans the split: per-request records (ctx,
//                     tiles, next request with tiles) and each CTA's first
//                     tile, balancing tiles plus a fixed cost per (b, h)
//                     segment a CTA starts (a segment start costs about as
//                     much as a few tiles: new Q, new masks, a drain of the
//                     MMA pipeline).
//   attn_tc_kernel    the append (an even share of the new rows per CTA,
//                     written while the first tiles load; tiles that reach
//                     the new positions take them from k_new / v_new) and
//                     the attention.  A (b, h) pair wholly inside one CTA
//                     writes its normalised output directly; a pair split
//                     over CTAs leaves one partial per CTA, and the CTA that
//                     completes the pair's tile count merges them by
//                     log-sum-exp.
//
// Per CTA, warp-specialised:
//   warps 10 and 7 (8 when R > 64)  producers: Q of each pair by TMA;
//               the K and V pages of each tile into a 4-stage ring (32 KB per
//               stage) by 16-byte cp.async copies placed in the swizzled
//               operand layout; the block ids of the next 32 tiles are
//               fetched one window ahead
//   warp 11     MMA issuer of S = Q K^T into TMEM (four buffers)
//   warp 9      MMA issuer of O += P V, P read back from TMEM (aliasing S);
//               two issuing threads because each tcgen05.mma takes about 90
//               cycles to issue, and one thread issuing both products of a
//               tile was the kernel's bottleneck
//   warps 0..7  softmax: one thread per query row (TMEM lane) and per half
//               tile (32 keys); each half reads the other half's scores too
//               for the tile maximum, so the two never wait for each other;
//               exp2, P written as bf16 into TMEM; O is rescaled in TMEM only
//               when the running maximum grows by more than 2^8; at a pair's
//               end, its output or partial
//
// TMEM: S0..S3 cols [0,64) .. [192,256), O [256,384), P0..P3 (bf16 pairs of
// S0..S3) [384,416) .. [480,512).  Four S buffers let Q K^T of tile t wait
// only for P V of tile t-4: the hand-off chain QK -> softmax -> PV -> QK of a
// buffer is spread over four tiles in flight (the K/V ring of four stages
// bounds the look-ahead to about three).  P has columns of its own so that
// no half ever writes over scores the other half is still reading.
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
constexpr int kCopyThreads = 64;    // threads issuing K/V copies (the copy warp and warp 10)
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
constexpr int kPCol = kOCol + 128;  // P of S buffer k (bf16 pairs) at kPCol + 32 k
// Split cost of one (request, head) segment, in tiles: the Q load, the
// masks and the drain of the pipeline at a pair's end cost about this much.
constexpr int kSegCost = 3;
constexpr int kPrepThreads = 256;
constexpr int kPlanReqs = 1024;  // requests whose plan arrays fit the prep kernel's shared memory

struct __align__(8) Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full[kQBufs];
  uint64_t q_empty[kQBufs];
  uint64_t s_full[kSBufs];
  uint64_t p_full[kSBufs];
  uint64_t o_done[kSBufs];  // completion of PV(t) lands on o_done[t % kSBufs]
  uint64_t drain[2];  // the Q K^T issuer's and the P V issuer's last completion
  uint64_t lbar[4];          // per sub-partition: both halves' row sums at a pair's output
  uint64_t ebar;             // every softmax warp wrote its rows of a partial
  float xl[2][128];          // [half][row] row sums at a pair's output
  uint32_t tmem_base;
  int abort;
  int tiles_issued[2];       // K/V tiles each copy warp issued (its loop may stop early)
};

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + kQBufs * kQBytes + sizeof(Bars) + 1024;

size_t smem_bytes() { return kSmemBytes; }

// Position in the flat tile sequence: request b, KV head h, tile of the
// pair, with the request's record (ctx, tiles per head, next request with
// tiles) and the next request's record loaded one request ahead, so that no
// role waits for a global load when it crosses into a new request.
struct Cursor {
  int b, h, tile, nt, ctx, next_b;
  int4 nrec;
  // st0 = (first tile, b, h, tile), st1 = (ctx, tiles, next request, end tile)
  __device__ void start(int4 st0, int4 st1, const int4* rq, int B) {
    b = st0.y;
    h = st0.z;
    tile = st0.w;
    ctx = st1.x;
    nt = st1.y;
    next_b = st1.z;
    nrec = make_int4(0, 0, B, 0);
    if (next_b < B) nrec = __ldcg(rq + next_b);
  }
  __device__ void next(const int4* rq, int B, int Hkv) {
    if (++tile < nt) return;
    tile = 0;
    if (++h < Hkv) return;
    h = 0;
    b = next_b;
    ctx = nrec.x;
    nt = nrec.y;
    next_b = nrec.z;
    if (next_b < B) nrec = __ldcg(rq + next_b);
  }
};

// Bits [s, s + 64) of the 128-bit mask (lo, hi) as one word, bit j holding
// mask bit s + j; bits outside [0, 128) read as 0 (s may be negative).
__device__ __forceinline__ unsigned long long mask_window(unsigned long long lo,
                                                          unsigned long long hi, int s) {
  if (s <= -64 || s >= 128) return 0ull;
  if (s < 0) return lo << -s;
  if (s == 0) return lo;
  if (s < 64) return (lo >> s) | (hi << (64 - s));
  return hi >> (s - 64);
}

// Keys of a tile visible to a row, bit j for tile column j: below the
// tile's valid keys and the request's length L, and either in the cached
// prefix (position < ctx) or a new position that is an ancestor-or-self of
// the row's node (bit pos - ctx of anc: up to 64 new rows).
__device__ __forceinline__ unsigned long long tile_visibility(int kpos0, int nkeys, int ctx, int L,
                                                              unsigned long long anc, bool real) {
  if (!real) return 0ull;
  const int lim = min(L - kpos0, nkeys);  // nkeys is 16..64
  unsigned long long v = lim >= 64 ? ~0ull : (lim <= 0 ? 0ull : ((1ull << lim) - 1));
  const int c0 = ctx - kpos0;  // tile columns in the cached prefix
  unsigned long long vm;
  if (c0 >= 64)
    vm = ~0ull;
  else if (c0 > 0)
    vm = ((1ull << c0) - 1) | (anc << c0);
  else
    vm = -c0 >= 64 ? 0ull : (anc >> -c0);
  return v & vm;
}

// The same for up to 128 new rows: the 128-bit mask (anc_lo, anc_hi).
__device__ __forceinline__ unsigned long long tile_visibility_wide(int kpos0, int nkeys, int ctx,
                                                                   int L, unsigned long long anc_lo,
                                                                   unsigned long long anc_hi,
                                                                   bool real) {
  if (!real) return 0ull;
  const int lim = min(L - kpos0, nkeys);  // nkeys is 16..64
  unsigned long long v = lim >= 64 ? ~0ull : (lim <= 0 ? 0ull : ((1ull << lim) - 1));
  const int c0 = ctx - kpos0;  // tile columns in the cached prefix
  const unsigned long long pre = c0 >= 64 ? ~0ull : (c0 > 0 ? ((1ull << c0) - 1) : 0ull);
  return v & (pre | mask_window(anc_lo, anc_hi, -c0));
}

// Ancestor-or-self mask of row i of a chain: bits 0..i.
__device__ __forceinline__ void chain_mask(int i, unsigned long long* lo, unsigned long long* hi) {
  *lo = i >= 63 ? ~0ull : ((1ull << (i + 1)) - 1);
  *hi = i >= 127 ? ~0ull : (i >= 64 ? ((1ull << (i - 63)) - 1) : 0ull);
}

__device__ __forceinline__ int tile_pages(int L, int tile) {
  const int keys = L - tile * kTileKeys;
  return keys >= kTileKeys ? kPages : ceil_div(keys, kBlock);
}

// 32 fp32 values (as bits) scaled and stored as bf16: a quarter row of out.
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                             float scale) {
#pragma unroll
  for (int j = 0; j < 32; j += 8) {
    uint4 w;
    w.x = ptx::pack_bf16x2(__uint_as_float(v[j]) * scale, __uint_as_float(v[j + 1]) * scale);
    w.y = ptx::pack_bf16x2(__uint_as_float(v[j + 2]) * scale, __uint_as_float(v[j + 3]) * scale);
    w.z = ptx::pack_bf16x2(__uint_as_float(v[j + 4]) * scale, __uint_as_float(v[j + 5]) * scale);
    w.w = ptx::pack_bf16x2(__uint_as_float(v[j + 6]) * scale, __uint_as_float(v[j + 7]) * scale);
    *reinterpret_cast<uint4*>(dst + j) = w;
  }
}

// kWide: more than 64 new rows per request (128-bit ancestor masks); the
// narrow kernel keeps one 64-bit word per row.  kShort: the wait limit is
// short (ptx::mbar_wait_t).
template <bool kWide, bool kShort>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* __restrict__ k_cache,
    __nv_bfloat16* __restrict__ v_cache, const int32_t* __restrict__ block_table,
    const int4* rq, const int4* starts, const ulonglong2* anc_ws, int* pairs, spec_dims d,
    float qscale2, float* part, __nv_bfloat16* __restrict__ out,
    float* __restrict__ lse, uint32_t* __restrict__ status) {
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
  const int c = blockIdx.x;
  const int n_sm_warps = ceil_div(R, 32);
  const uint64_t wait = wait_limit_cycles(d);
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
    for (int sp = 0; sp < 4; ++sp) ptx::mbar_init(ptx::smem_u32(&bars->lbar[sp]), 2);
    ptx::mbar_init(ptx::smem_u32(&bars->ebar), 2 * n_sm_warps);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) ptx::prefetch_tmap(&tm_q);
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;

  pdl_wait();  // the plan comes from the previous kernel
  const int4 st0 = __ldcg(starts + 2 * c), st1 = __ldcg(starts + 2 * c + 1);
  const int64_t g0 = st0.x, g1 = st1.w;
  const bool idle = g0 >= g1;  // uniform: no tiles for this CTA
  const int copy_warp = n_sm_warps <= 2 ? kCopyWarpSmallR : kCopyWarpLargeR;

  // ------------------------------------------------------------------ append
  // The new rows go into the cache while the first tiles load: every CTA
  // writes an even share of all (request, position, head, 16-byte chunk)
  // items, positions ctx .. end-1 with end = ceil(L/16)*16 (rows past
  // ctx+M-1 cleared).  The attention itself reads the new rows from
  // k_new / v_new, so nothing waits for these writes.  Writers: every thread
  // of a CTA without tiles, else the warps without a role (softmax warps of
  // padding sub-partitions, warp 8 when warp 7 copies), else, when R > 96
  // leaves none, the softmax warps before their first tile.
  uint32_t writers = 0;  // bit w: warp w writes
  for (int w = 0; w <= kCopyWarpLargeR; ++w)
    if (w != copy_warp && (w >= kSoftmaxWarps || (w & 3) >= n_sm_warps)) writers |= 1u << w;
  if (writers == 0) writers = ((1u << kSoftmaxWarps) - 1) & ~(1u << copy_warp);
  if (idle) writers = (1u << (kThreads / kWarp)) - 1;
  if ((writers >> warp) & 1u) {
    const int nthr = __popc(writers) * kWarp;
    const int wtid = __popc(writers & ((1u << warp) - 1)) * kWarp + lane;
    const int per_pos = Hkv * 16;  // items of one position (D = 128)
    const int per_req = (M + kBlock - 1) * per_pos;
    const int64_t n_items = (int64_t)B * per_req;
    const int64_t i0 = (int64_t)c * n_items / gridDim.x, i1 = (int64_t)(c + 1) * n_items / gridDim.x;
#pragma unroll 2
    for (int64_t it = i0 + wtid; it < i1; it += nthr) {
      const int b = (int)(it / per_req);
      const int rem = (int)(it - (int64_t)b * per_req);
      const int pi = rem / per_pos;
      const int h = (rem / 16) % Hkv;
      const int ch = rem % 16;
      const int4 r = __ldcg(rq + b);  // (ctx, tiles, ...): no tiles means the request failed its checks
      const int64_t tpos = (int64_t)r.x + pi;
      if (r.y == 0 || tpos >= ceil_div64((int64_t)r.x + M, kBlock) * kBlock) continue;
      const int64_t dst = (((int64_t)block_table[(int64_t)b * d.max_blocks + tpos / kBlock] * Hkv + h) *
                               kBlock + tpos % kBlock) * 128 + ch * 8;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (pi < M) {
        const int64_t src = (((int64_t)b * M + pi) * Hkv + h) * 128 + ch * 8;
        kv = *reinterpret_cast<const uint4*>(k_new + src);
        vv = *reinterpret_cast<const uint4*>(v_new + src);
      }
      *reinterpret_cast<uint4*>(k_cache + dst) = kv;
      *reinterpret_cast<uint4*>(v_cache + dst) = vv;
    }
  }
  if (idle) {
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
    return;
  }
  // Only a CTA's first segment can be a later share of a split pair (it
  // starts inside the pair).  Its tiles are counted for the merging CTA by a
  // warp without a role, after the softmax warps have written the partial,
  // so that the fence before the count stalls no softmax warp.
  const int helper = n_sm_warps <= 2 ? kCopyWarpLargeR : (n_sm_warps == 3 ? 3 : -1);
  if (warp == helper && lane == 0 && st0.w > 0) {
    if (ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->ebar), 0, abort, wait)) {
      __threadfence();
      atomicAdd(pairs + (int64_t)st0.y * Hkv + st0.z, (int)min((int64_t)(st1.y - st0.w), g1 - g0));
    }
  }

  if (warp == kProducerWarp || warp == copy_warp) {
    // ------------------------------------------------------------ producers
    // Both warps walk the tiles; lane j holds the four block ids of tile
    // (window start + j) of a window of 32 tiles, and the ids of the next
    // window are loaded when a window starts.  Q comes by TMA (warp 10,
    // lane 0).  K and V come by 16-byte cp.async copies from all 64
    // threads, each placed where the 128-byte-swizzled layout of the MMA
    // operands wants it (chunk j of row r of a page at j ^ (r % 8)): one
    // tensor-TMA box per page half bounded the kernel at about 16 boxes per
    // tile, whatever their size.
    const int ct = (warp == copy_warp ? 0 : kWarp) + lane;  // copy thread 0..63
    const int c16 = ct & 15;                                 // 16-byte chunk of a 256-byte row
    const int r0 = ct >> 4;                                  // rows r0, r0 + 4, r0 + 8, r0 + 12
    const uint32_t swz_half = (uint32_t)(c16 >> 3) * kHalfBytes;
    Cursor cu;
    cu.start(st0, st1, rq, B);
    int seg = -1, L = 0;
    int wb = -1, ww = -1, nb = -1, nw = -1;  // window held in ids and window loaded into nids
    int ids[kPages] = {0, 0, 0, 0}, nids[kPages] = {0, 0, 0, 0};
    int64_t t = 0;
    int q_issued = 0;  // Q loads issued (warp 10, lane 0)
    bool ok = true;
    for (int64_t g = g0; g < g1 && ok; ++g, ++t) {
      const bool first = (g == g0) || cu.tile == 0;
      if (first) {
        ++seg;
        L = cu.ctx + M;
        if (warp == kProducerWarp) {
          if (lane == 0) {
            const int qb = seg % kQBufs;
            ok = ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->q_empty[qb]), ((seg / kQBufs) & 1) ^ 1, abort,
                                wait);
            if (ok) {
              const uint32_t qf = ptx::smem_u32(&bars->q_full[qb]);
              ptx::mbar_arrive_expect_tx(qf, 2u * R * 128u);
              for (int half = 0; half < 2; ++half)
                ptx::tma_load_4d(ptx::smem_u32(qbufs + qb * kQBytes + half * kQBytes / 2), &tm_q,
                                 qf, half * 64, cu.h * group, 0, cu.b);
              ++q_issued;
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
      }
      const int w = cu.tile >> 5;
      if (cu.b != wb || w != ww) {  // next window of 32 tiles
        if (cu.b == nb && w == nw) {
#pragma unroll
          for (int p = 0; p < kPages; ++p) ids[p] = nids[p];
        } else {
          const int page0 = ((w << 5) + lane) * kPages;
          const int32_t* bt = block_table + (int64_t)cu.b * d.max_blocks;
#pragma unroll
          for (int p = 0; p < kPages; ++p) ids[p] = (page0 + p < d.max_blocks) ? bt[page0 + p] : 0;
        }
        wb = cu.b;
        ww = w;
        // the next window with other ids: the pair's next window, else the
        // first of the next head (same ids when the pair has one window:
        // then the next request's first)
        if ((w + 1) * 32 < cu.nt) {
          nb = cu.b;
          nw = w + 1;
        } else {
          nb = (cu.h + 1 < Hkv && w > 0) ? cu.b : cu.next_b;
          nw = 0;
        }
        if (nb == wb && nw == ww) {
#pragma unroll
          for (int p = 0; p < kPages; ++p) nids[p] = ids[p];
        } else if (nb < B) {
          const int page0 = ((nw << 5) + lane) * kPages;
          const int32_t* bt = block_table + (int64_t)nb * d.max_blocks;
#pragma unroll
          for (int p = 0; p < kPages; ++p) nids[p] = (page0 + p < d.max_blocks) ? bt[page0 + p] : 0;
        }
      }
      const int np = tile_pages(L, cu.tile);
      const int src = cu.tile & 31;
      int blk[kPages];
#pragma unroll
      for (int p = 0; p < kPages; ++p) blk[p] = __shfl_sync(0xffffffffu, ids[p], src);
      const int stage = (int)(t % kStages);
      ok = ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->empty[stage]), (uint32_t)((t / kStages) & 1) ^ 1u,
                          abort, wait);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint32_t sb = ptx::smem_u32(stages + stage * kStageBytes);
      const int kpos0 = cu.tile * kTileKeys;
      if (kpos0 + kTileKeys <= cu.ctx) {  // all keys in the cached prefix
#pragma unroll
        for (int p = 0; p < kPages; ++p) {
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
      } else {
        // the tile reaches the new rows: those come from k_new / v_new (the
        // append into the cache runs concurrently), rows past L are zero
#pragma unroll
        for (int p = 0; p < kPages; ++p) {
          if (p < np) {
            const int64_t page = ((int64_t)blk[p] * Hkv + cu.h) * kBlock;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int r = r0 + 4 * k;
              const int pos = kpos0 + p * kBlock + r;
              const uint32_t so = swz_half + (uint32_t)p * kBoxBytes + (uint32_t)r * 128u +
                                  ((uint32_t)((c16 & 7) ^ (r & 7)) << 4);
              if (pos < cu.ctx) {
                const int64_t e = (page + r) * 128 + c16 * 8;
                ptx::cp_async16(sb + so, k_cache + e);
                ptx::cp_async16(sb + 2 * kHalfBytes + so, v_cache + e);
              } else {
                const bool in = pos < L;
                const int64_t e = in ? (((int64_t)cu.b * M + (pos - cu.ctx)) * Hkv + cu.h) * 128 + c16 * 8 : 0;
                ptx::cp_async16_fill(sb + so, k_new + e, in ? 16u : 0u);
                ptx::cp_async16_fill(sb + 2 * kHalfBytes + so, v_new + e, in ? 16u : 0u);
              }
            }
          }
        }
      }
      ptx::cp_async_arrive_noinc(ptx::smem_u32(&bars->full[stage]));
      cu.next(rq, B, Hkv);
    }
    // Every copy issued lands before the CTA may exit, also when a wait gave
    // up and the two copy warps stopped at different tiles: each thread's
    // own cp.async copies (wait_all), then the full barriers of the tiles
    // both warps issued (their arrivals follow the copies), then the Q loads
    // actually issued.  A barrier that only one warp arrived on is never
    // waited for.
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0) bars->tiles_issued[warp == kProducerWarp ? 1 : 0] = (int)t;
    asm volatile("bar.sync 1, 64;" ::: "memory");  // the two copy warps only
    if (warp == kProducerWarp && lane == 0) {
      const int64_t both = min(bars->tiles_issued[0], bars->tiles_issued[1]);
      for (int64_t u = both > kStages ? both - kStages : 0; u < both; ++u)
        ptx::mbar_drain(ptx::smem_u32(&bars->full[u % kStages]), (uint32_t)((u / kStages) & 1),
                        kDefaultWaitCycles);
      for (int sg = q_issued > kQBufs ? q_issued - kQBufs : 0; sg < q_issued; ++sg)
        ptx::mbar_drain(ptx::smem_u32(&bars->q_full[sg % kQBufs]), (uint32_t)((sg / kQBufs) & 1),
                        kDefaultWaitCycles);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA: Q K^T
    if (lane == 0) {
      const uint32_t id_qk_full = ptx::idesc_bf16_f32(128, kTileKeys, false, false);
      Cursor cu;
      cu.start(st0, st1, rq, B);
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
        if (first) {
          ++seg;
          L = cu.ctx + M;
        }
        const int qb = seg % kQBufs;
        if (first && !ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->q_full[qb]),
                                     (uint32_t)((seg / kQBufs) & 1), abort, wait))
          break;
        const int stage = (int)(t % kStages);
        if (!ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->full[stage]), (uint32_t)((t / kStages) & 1),
                            abort, wait))
          break;
        // PV(t - kSBufs) read P out of the S buffer this tile's QK writes
        if (t >= kSBufs && !ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->o_done[t % kSBufs]),
                                           (uint32_t)(((t - kSBufs) / kSBufs) & 1), abort,
                                           wait))
          break;
        ptx::tc_fence_after();
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
        cu.next(rq, B, Hkv);
      }
      // all MMAs issued by this thread complete before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&bars->drain[0]));
      ptx::mbar_drain(ptx::smem_u32(&bars->drain[0]), 0, kDefaultWaitCycles);
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
      cu.start(st0, st1, rq, B);
      int L = 0;
      int64_t u = 0;
      for (int64_t g = g0; g < g1; ++g, ++u) {
        const bool first = (g == g0) || cu.tile == 0;
        if (first) L = cu.ctx + M;
        const int np = tile_pages(L, cu.tile);
        const int sbuf = (int)(u % kSBufs);
        const int stage = (int)(u % kStages);
        if (!ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->p_full[sbuf]), (uint32_t)((u / kSBufs) & 1), abort,
                            wait))
          break;
        ptx::tc_fence_after();
        const uint64_t dv = dv0 + (uint64_t)((stage * kStageBytes) >> 4);
        const uint32_t pcol = tmem + kPCol + sbuf * 32;
#pragma unroll
        for (int j = 0; j < kPages; ++j) {
          if (j < np)
            ptx::mma_ts(tmem + kOCol, pcol + j * 8, dv + (uint64_t)((j * 2 * 1024) >> 4), id_pv,
                        (first && j == 0) ? 0u : 1u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->o_done[sbuf]));
        ptx::mma_commit(ptx::smem_u32(&bars->empty[stage]));
        cu.next(rq, B, Hkv);
      }
      ptx::mma_commit(ptx::smem_u32(&bars->drain[1]));
      ptx::mbar_drain(ptx::smem_u32(&bars->drain[1]), 0, kDefaultWaitCycles);
    }
  } else if (warp < kSoftmaxWarps) {
    // -------------------------------------------------------------- softmax
    const int sp = warp & 3;   // TMEM sub-partition this warp may access
    const int half = warp >> 2;  // keys [32*half, 32*half + 32) of each tile
    const int row = sp * 32 + lane;
    if (sp < n_sm_warps) {
      const uint32_t lane_base = tmem + ((uint32_t)(sp * 32) << 16);
      const int S = tc_part_stride(d.D);
      Cursor cu;
      cu.start(st0, st1, rq, B);
      int64_t t = 0;
      float m_used = -INFINITY, l = 0.f;
      unsigned long long anc = 0, anc_n = 0;        // mask bits 0..63
      unsigned long long anc_hi = 0, anc_hi_n = 0;  // bits 64..127 (kWide)
      int anc_b = -1, anc_nb = -1;  // requests whose masks anc and anc_n hold
      int ctx = 0, L = 0, tile0 = 0;
      int n_whole = 0;  // pair ends with output so far (barrier phase)
      const bool real = row < R;
      const int i = real ? row / group : 0;
      for (int64_t g = g0; g < g1; ++g, ++t) {
        const bool first = (g == g0) || cu.tile == 0;
        const bool last = (g == g1 - 1) || cu.tile == cu.nt - 1;
        if (first) {
          ctx = cu.ctx;
          L = ctx + M;
          tile0 = cu.tile;
          m_used = -INFINITY;
          l = 0.f;
          if (anc_ws == nullptr) {
            if (kWide) chain_mask(i, &anc, &anc_hi);
            else anc = (i >= 63) ? ~0ull : ((1ull << (i + 1)) - 1);
          } else if (real && cu.b != anc_b) {
            // tree masks come from the prep kernel; the next request's mask
            // is loaded one request ahead
            const unsigned long long* aw = reinterpret_cast<const unsigned long long*>(anc_ws);
            if (cu.b == anc_nb) {
              anc = anc_n;
              if (kWide) anc_hi = anc_hi_n;
            } else {
              anc = __ldcg(aw + 2 * ((int64_t)cu.b * M + i));
              if (kWide) anc_hi = __ldcg(aw + 2 * ((int64_t)cu.b * M + i) + 1);
            }
            anc_b = cu.b;
            if (cu.next_b < B) {
              anc_n = __ldcg(aw + 2 * ((int64_t)cu.next_b * M + i));
              if (kWide) anc_hi_n = __ldcg(aw + 2 * ((int64_t)cu.next_b * M + i) + 1);
              anc_nb = cu.next_b;
            }
          }
        }
        const int sbuf = (int)(t % kSBufs);  // S / P buffer in TMEM
        if (!__all_sync(0xffffffffu, ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->s_full[sbuf]),
                                                     (uint32_t)((t / kSBufs) & 1), abort, wait)))
          break;
        ptx::tc_fence_after();
        const int kpos0 = cu.tile * kTileKeys;
        const int nkeys = tile_pages(L, cu.tile) * kBlock;
        // tiles wholly inside the cached prefix need no mask
        const bool plain = kpos0 + kTileKeys <= ctx && nkeys == kTileKeys;
        const int jbase = half * 32;
        uint32_t vh = 0xffffffffu;  // visible keys of this half (non-plain tiles)
        uint32_t sv[32], so[32];
        ptx::tmem_ld32(lane_base + sbuf * kTileKeys + jbase, sv);
        ptx::tmem_ld32(lane_base + sbuf * kTileKeys + (jbase ^ 32), so);
        ptx::tmem_wait_ld();
        // maximum of the whole tile (log2 units): this half's columns and the
        // other half's, read straight from TMEM, so that both halves reach
        // the same maximum without waiting for each other (P goes to its own
        // columns, never over S)
        float mt;
        if (plain) {
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            a0 = fmaxf(a0, __uint_as_float(sv[j]));
            a1 = fmaxf(a1, __uint_as_float(sv[j + 1]));
            a2 = fmaxf(a2, __uint_as_float(sv[j + 2]));
            a3 = fmaxf(a3, __uint_as_float(sv[j + 3]));
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            a0 = fmaxf(a0, __uint_as_float(so[j]));
            a1 = fmaxf(a1, __uint_as_float(so[j + 1]));
            a2 = fmaxf(a2, __uint_as_float(so[j + 2]));
            a3 = fmaxf(a3, __uint_as_float(so[j + 3]));
          }
          mt = real ? fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * qscale2 : -INFINITY;
        } else {
          // visibility of the tile's keys as a bitmask, then the same maximum
          // as the plain path over the visible ones
          const unsigned long long vis =
              kWide ? tile_visibility_wide(kpos0, nkeys, ctx, L, anc, anc_hi, real)
                    : tile_visibility(kpos0, nkeys, ctx, L, anc, real);
          vh = (uint32_t)(vis >> jbase);
          const uint32_t vo = (uint32_t)(vis >> (jbase ^ 32));
          float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            a0 = fmaxf(a0, (vh >> j) & 1u ? __uint_as_float(sv[j]) : -INFINITY);
            a1 = fmaxf(a1, (vh >> (j + 1)) & 1u ? __uint_as_float(sv[j + 1]) : -INFINITY);
          }
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            a0 = fmaxf(a0, (vo >> j) & 1u ? __uint_as_float(so[j]) : -INFINITY);
            a1 = fmaxf(a1, (vo >> (j + 1)) & 1u ? __uint_as_float(so[j + 1]) : -INFINITY);
          }
          mt = fmaxf(a0, a1) * qscale2;
        }
        bool need = false;
        if (first) {
          m_used = mt;
        } else if (mt > m_used + 8.0f) {
          need = true;
        }
        if (__any_sync(0xffffffffu, need)) {
          // O is rescaled in place (this half's 64 columns): PV(t-1) must have landed
          if (!__all_sync(0xffffffffu,
                          ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->o_done[(t - 1) % kSBufs]),
                                         (uint32_t)(((t - 1) / kSBufs) & 1), abort, wait)))
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
        // probabilities of this half, packed to bf16 pairs: keys 32*half..
        // land in columns 16*half.. of the buffer's P columns
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
          const float nm = -m_used;  // finite whenever a key of the row is visible
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float pa = (vh >> (2 * j)) & 1u
                                 ? fast_exp2(fmaf(__uint_as_float(sv[2 * j]), qscale2, nm))
                                 : 0.f;
            const float pb = (vh >> (2 * j + 1)) & 1u
                                 ? fast_exp2(fmaf(__uint_as_float(sv[2 * j + 1]), qscale2, nm))
                                 : 0.f;
            l0 += pa;
            l1 += pb;
            pk[j] = ptx::pack_bf16x2(pa, pb);
          }
        }
        l += l0 + l1;
        ptx::tmem_st16(lane_base + kPCol + sbuf * 32 + half * 16, pk);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full[sbuf]));
        if (last) {
          if (!__all_sync(0xffffffffu, ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->o_done[sbuf]),
                                                       (uint32_t)((t / kSBufs) & 1), abort, wait)))
            break;
          ptx::tc_fence_after();
          const int64_t pair = (int64_t)cu.b * Hkv + cu.h;
          const int hq = cu.h * group + (real ? row % group : 0);
          __nv_bfloat16* orow = out + (((int64_t)cu.b * M + i) * d.Hq + hq) * d.D + half * 64;
          float* lrow = lse != nullptr ? lse + ((int64_t)cu.b * M + i) * d.Hq + hq : nullptr;
          const int own = cu.tile - tile0 + 1;  // tiles of the pair run by this CTA
          if (tile0 > 0) {
            // ---- a later share of a split pair: a partial for the CTA that
            // ran the pair's first tile (unnormalised O of this half's 64
            // columns, the running maximum, this half's row sum, the tiles)
            float* prow = part + ((pair + c) * R + (real ? row : 0)) * (int64_t)S;
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
              if (half == 0) {
                prow[d.D] = m_used;
                prow[d.D + 3] = __int_as_float(own);
              }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ebar));
            if (helper < 0 && warp == 0 && lane == 0 &&
                ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->ebar), 0, abort, wait)) {
              // every row of the partial is written (the barrier above); the
              // fence makes them visible GPU-wide before the tiles are counted
              __threadfence();
              atomicAdd(pairs + pair, own);
            }
          } else {
            // ---- the pair's first CTA: its own rows from TMEM, merged with
            // the partials of the CTAs that ran the rest of the pair (none
            // when the whole pair ran here)
            bars->xl[half][row] = l;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->lbar[sp]));
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_t<kShort>(ptx::smem_u32(&bars->lbar[sp]),
                                                         (uint32_t)(n_whole & 1), abort, wait)))
              break;
            ++n_whole;
            float ls = bars->xl[0][row] + bars->xl[1][row];
            float mx = m_used;
            const int rest = cu.nt - own;  // tiles run by the CTAs after this one
            bool okc = true;
            if (rest > 0) {
              if (lane == 0) okc = ptx::wait_count_geq(pairs + pair, rest, abort, wait);
              __syncwarp();
              okc = __shfl_sync(0xffffffffu, okc, 0);
            }
            if (!okc) break;
            // Two passes over this half's 64 columns, 32 at a time.  Each walks
            // up from CTA c+1 until the partials' tiles add up (CTAs with no
            // tiles, possible when there are more CTAs than split costs, wrote
            // nothing), loading a partial's scalars with its columns.  The
            // first pass also finds the common maximum and the row sum; the
            // second reuses them.
            const float m_own = m_used;
#pragma unroll 1
            for (int cc2 = 0; cc2 < 2; ++cc2) {
              uint32_t o[32];
              ptx::tmem_ld32(lane_base + kOCol + half * 64 + cc2 * 32, o);
              ptx::tmem_wait_ld();
              // o holds sum w * O relative to the maximum mx; in the first pass
              // mx grows as partials come in, in the second it is final
              const float w_own = cc2 == 0 ? 1.f : (m_own == -INFINITY ? 0.f : exp2f(m_own - mx));
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * w_own);
              for (int got = 0, cq = c + 1; got < rest && cq < (int)gridDim.x; ++cq) {
                const int ga = __ldcg(&starts[2 * cq].x), gb = __ldcg(&starts[2 * cq + 1].w);
                const float* q = part + ((pair + cq) * R + (real ? row : 0)) * (int64_t)S;
                const float4 sc = __ldcg(reinterpret_cast<const float4*>(q + d.D));
                float4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  v[j] = __ldcg(reinterpret_cast<const float4*>(q + half * 64 + cc2 * 32) + j);
                if (ga == gb) continue;
                got += __float_as_int(sc.w);
                const float lq = sc.y + sc.z;
                if (!(lq > 0.f)) continue;
                float a = 1.f, w;
                if (cc2 == 0) {
                  const float mn = fmaxf(mx, sc.x);
                  a = mx == -INFINITY ? 0.f : exp2f(mx - mn);
                  w = exp2f(sc.x - mn);
                  ls = ls * a + lq * w;
                  mx = mn;
                } else {
                  w = exp2f(sc.x - mx);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  o[4 * j] = __float_as_uint(fmaf(w, v[j].x, a * __uint_as_float(o[4 * j])));
                  o[4 * j + 1] = __float_as_uint(fmaf(w, v[j].y, a * __uint_as_float(o[4 * j + 1])));
                  o[4 * j + 2] = __float_as_uint(fmaf(w, v[j].z, a * __uint_as_float(o[4 * j + 2])));
                  o[4 * j + 3] = __float_as_uint(fmaf(w, v[j].w, a * __uint_as_float(o[4 * j + 3])));
                }
              }
              if (real) store32_bf16(orow + cc2 * 32, o, ls > 0.f ? 1.f / ls : 0.f);
            }
            if (real && half == 0 && lrow != nullptr)
              *lrow = ls > 0.f ? (mx + log2f(ls)) * 0.69314718055994530942f : -INFINITY;
          }
          ptx::tc_fence_before();
        }
        cu.next(rq, B, Hkv);
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
// request checks and the plan of the split
// ---------------------------------------------------------------------------
// Exclusive prefix over the CTA's threads of two int64 sums and an int max.
__device__ __forceinline__ void block_scan(int64_t& a, int64_t& c, int& m, int64_t* sa,
                                           int64_t* sc, int* sm, int64_t& ta, int64_t& tc_,
                                           int& tm) {
  const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
  const int nw = blockDim.x / kWarp;
  int64_t ia = a, ic = c;
  int im = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t ya = __shfl_up_sync(0xffffffffu, ia, o);
    const int64_t yc = __shfl_up_sync(0xffffffffu, ic, o);
    const int ym = __shfl_up_sync(0xffffffffu, im, o);
    if (lane >= o) {
      ia += ya;
      ic += yc;
      im = max(im, ym);
    }
  }
  if (lane == 31) {
    sa[warp] = ia;
    sc[warp] = ic;
    sm[warp] = im;
  }
  __syncthreads();
  int64_t pa = 0, pc = 0;
  int pm = -1;
  for (int w = 0; w < warp; ++w) {
    pa += sa[w];
    pc += sc[w];
    pm = max(pm, sm[w]);
  }
  ta = tc_ = 0;
  tm = -1;
  for (int w = 0; w < nw; ++w) {
    ta += sa[w];
    tc_ += sc[w];
    tm = max(tm, sm[w]);
  }
  // exclusive values: the prefix of the earlier warps plus the lanes before
  const int xm = __shfl_up_sync(0xffffffffu, im, 1);
  a = pa + ia - a;
  c = pc + ic - c;
  m = max(pm, lane > 0 ? xm : -1);
  __syncthreads();
}

// One CTA per request.  Checks the request (capacity, the block ids of every
// page it reads or writes, the tree topology) and records it for the plan.
// A request that fails gets out = 0, lse = -inf and no tiles (the attention
// kernel then neither reads nor appends it).  The CTA that arrives last
// plans the split of the tiles.
__global__ void __launch_bounds__(kPrepThreads) attn_prep_kernel(
    const int32_t* block_table, const int32_t* ctx_lens,
    const int32_t* __restrict__ parent, spec_dims d, int G, int32_t* __restrict__ ntiles,
    int64_t* __restrict__ pre, int4* __restrict__ rq, int4* __restrict__ starts,
    int* __restrict__ pairs, ulonglong2* __restrict__ anc_ws,
    uint32_t* __restrict__ arrivals, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
    uint32_t* __restrict__ status) {
  __shared__ int s_last;
  __shared__ int64_t s_a[kPrepThreads / kWarp], s_c[kPrepThreads / kWarp];
  __shared__ int s_m[kPrepThreads / kWarp];
  // the plan's working arrays (used by the last CTA only)
  __shared__ int64_t s_tpre[kPlanReqs + 1], s_cpre[kPlanReqs + 1];
  __shared__ int s_nt[kPlanReqs], s_ctx[kPlanReqs], s_next[kPlanReqs];
  __shared__ int s_g0[kMaxAttnCtas + 1], s_req[kMaxAttnCtas];
  pdl_trigger();
  pdl_wait();  // the inputs and the cache may come from the previous kernel
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int B = d.B, M = d.M, Hkv = d.Hkv, D = d.D;
  const int32_t* bt = block_table + (int64_t)b * d.max_blocks;
  // The table's first kPrepPages * kPrepThreads entries are loaded together
  // with the context length (all in bounds of the table), so the check does
  // not wait for the length before its loads.
  constexpr int kPrepPages = 8;
  int ids[kPrepPages];
#pragma unroll
  for (int k = 0; k < kPrepPages; ++k) {
    const int p = tid + k * kPrepThreads;
    ids[k] = p < d.max_blocks ? __ldcg(bt + p) : 0;
  }
  const int ctx = __ldcg(ctx_lens + b);
  const int64_t L = (int64_t)ctx + M;
  const int64_t cap = (int64_t)d.max_blocks * kBlock;

  const bool cap_ok = ctx >= 0 && L <= cap;
  int bad_block = 0;
  if (cap_ok) {
    const int pages = (int)ceil_div64(L, kBlock);
#pragma unroll
    for (int k = 0; k < kPrepPages; ++k)
      if (tid + k * kPrepThreads < pages) bad_block |= (ids[k] < 0 || ids[k] >= d.num_blocks);
#pragma unroll 4
    for (int p = tid + kPrepPages * kPrepThreads; p < pages; p += kPrepThreads) {
      const int id = __ldcg(bt + p);
      bad_block |= (id < 0 || id >= d.num_blocks);
    }
  }
  int bad_topo = 0;
  if (parent != nullptr) {
    const int32_t* par = parent + (int64_t)b * M;
    for (int n = tid; n < M; n += blockDim.x) {
      const int pn = par[n];
      bad_topo |= (n == 0) ? (pn != -1) : (pn < 0 || pn >= n);
    }
  }
  bad_block = __syncthreads_or(bad_block);
  bad_topo = __syncthreads_or(bad_topo);
  const bool ok = cap_ok && !bad_block && !bad_topo;
  // tile counts of the request's (request, head) pairs start at zero
  for (int h = tid; h < Hkv; h += blockDim.x) pairs[(int64_t)b * Hkv + h] = 0;
  if (ok && parent != nullptr) {
    // ancestor-or-self mask of each tree row (the topology is valid here,
    // so every walk ends at the root within M steps)
    const int32_t* par = parent + (int64_t)b * M;
    for (int n = tid; n < M; n += blockDim.x) {
      unsigned long long lo = 0, hi = 0;  // bits 0..63, 64..127
      for (int k = n; k >= 0; k = par[k]) {
        if (k < 64) lo |= 1ull << k;
        else hi |= 1ull << (k - 64);
      }
      anc_ws[(int64_t)b * M + n] = make_ulonglong2(lo, hi);
    }
  }
  if (tid == 0) {
    if (!cap_ok) raise_status(status, SPEC_ERR_CAPACITY);
    if (bad_block) raise_status(status, SPEC_ERR_DEVICE_BOUNDS);
    if (bad_topo) raise_status(status, SPEC_ERR_INVALID_ARG);
    ntiles[b] = ok ? (int)ceil_div64(L, kTileKeys) : 0;
    __threadfence();
    s_last = atomicAdd(arrivals, 1u) == (uint32_t)(B - 1);
  }
  __syncthreads();

  if (!ok) {
    const int lanes = D / 8;  // 16-byte vectors per (position, head)
    const int64_t n = (int64_t)M * d.Hq * lanes;
    for (int64_t w = tid; w < n; w += blockDim.x)
      reinterpret_cast<uint4*>(out + (int64_t)b * M * d.Hq * D)[w] = make_uint4(0, 0, 0, 0);
    if (lse != nullptr)
      for (int w = tid; w < M * d.Hq; w += blockDim.x) lse[(int64_t)b * M * d.Hq + w] = -INFINITY;
  }
  if (!s_last) return;

  // ---- the plan, by the last CTA to arrive.  Request r costs
  // Hkv * (tiles + kSegCost) when it has tiles; a pair's fixed cost comes
  // before its first tile, so tile j of a pair starts at cost
  // base + kSegCost + j, and CTA k starts at the first tile whose cost
  // reaches k * total / G.
  __threadfence();
  // Up to kPlanReqs requests the plan's per-request arrays live in shared
  // memory (no global round trips after the first load), beyond that in the
  // workspace.
  const bool small = B <= kPlanReqs;
  int64_t* tpre = small ? s_tpre : pre;          // [B+1] tiles before request r
  int64_t* cpre = small ? s_cpre : pre + B + 1;  // [B+1] split cost before request r
  int64_t carry_t = 0, carry_c = 0;
  int carry_m = -1;
  for (int base = 0; base < B; base += blockDim.x) {
    const int r = base + tid;
    const int nt = r < B ? __ldcg(ntiles + r) : 0;
    const int cx = r < B ? ctx_lens[r] : 0;
    int64_t vt = (int64_t)nt * Hkv, vc = nt > 0 ? (int64_t)Hkv * (nt + kSegCost) : 0;
    int vm = nt > 0 ? r : -1;
    int64_t tt, tcst;
    int tm;
    block_scan(vt, vc, vm, s_a, s_c, s_m, tt, tcst, tm);
    const int prev = max(vm, carry_m);  // the last request with tiles before r
    if (r < B) {
      tpre[r] = carry_t + vt;
      cpre[r] = carry_c + vc;
      rq[r] = make_int4(cx, nt, B, 0);
      if (small) {
        s_nt[r] = nt;
        s_ctx[r] = cx;
        s_next[r] = B;
      }
    }
    __syncthreads();
    if (r < B && nt > 0 && prev >= 0) {
      reinterpret_cast<int*>(rq + prev)[2] = r;
      if (small) s_next[prev] = r;
    }
    carry_t += tt;
    carry_c += tcst;
    carry_m = max(carry_m, tm);
    __syncthreads();
  }
  const int64_t T = carry_t, Ctot = carry_c;
  if (tid == 0) {
    tpre[B] = T;
    cpre[B] = Ctot;
    starts[2 * G] = make_int4((int)T, B, 0, 0);
    starts[2 * G + 1] = make_int4(0, 0, B, (int)T);
    s_g0[G] = (int)T;
    *arrivals = 0;
  }
  __syncthreads();
  if (Ctot == 0) {
    for (int k = tid; k < G; k += blockDim.x) {
      starts[2 * k] = make_int4(0, B, 0, 0);
      starts[2 * k + 1] = make_int4(0, 0, B, 0);
    }
    return;
  }
  for (int r = tid; r < B; r += blockDim.x) {
    const int64_t c0 = cpre[r], c1 = cpre[r + 1];
    if (c1 == c0) continue;
    const int nt = small ? s_nt[r] : __ldcg(ntiles + r);
    const int64_t per = nt + kSegCost;
    // CTAs k with c0 <= floor(k * Ctot / G) < c1
    const int k0 = (int)((c0 * G + Ctot - 1) / Ctot), k1 = (int)((c1 * G + Ctot - 1) / Ctot);
    for (int k = k0; k < k1; ++k) {
      int64_t rem = (int64_t)k * Ctot / G - c0;
      const int h = (int)(rem / per);
      rem -= h * per;
      const int j = (int)max((int64_t)0, rem - kSegCost);  // rem < nt + kSegCost: j < nt
      const int g0 = (int)(tpre[r] + (int64_t)h * nt + j);
      starts[2 * k] = make_int4(g0, r, h, j);
      s_g0[k] = g0;
      s_req[k] = r;
    }
  }
  __syncthreads();
  // second half of each start record: the first request's record and the
  // CTA's end tile (a CTA with tiles starts inside a request)
  for (int k = tid; k < G; k += blockDim.x) {
    const int r = s_req[k];
    const int4 rec = small ? make_int4(s_ctx[r], s_nt[r], s_next[r], 0) : rq[r];
    starts[2 * k + 1] = make_int4(rec.x, rec.y, rec.z, s_g0[k + 1]);
  }
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
  // flat tile indices are int32: every request's tiles of every head
  if ((int64_t)d.B * d.Hkv * ceil_div64((int64_t)d.max_blocks * kBlock, kTileKeys) > INT32_MAX)
    return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.ws);
  int32_t* ntiles = reinterpret_cast<int32_t*>(ws + lay.tc_ntiles_off);
  int64_t* pre = reinterpret_cast<int64_t*>(ws + lay.tc_pre_off);
  int4* rq = reinterpret_cast<int4*>(ws + lay.tc_rq_off);
  int4* starts = reinterpret_cast<int4*>(ws + lay.tc_start_off);
  int* pairs = reinterpret_cast<int*>(ws + lay.tc_pair_off);
  ulonglong2* anc = reinterpret_cast<ulonglong2*>(ws + lay.tc_anc_off);
  uint32_t* arrivals = reinterpret_cast<uint32_t*>(ws + lay.tc_sync_off);
  float* part = reinterpret_cast<float*>(ws + lay.attn_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + lay.status_off);

  CUtensorMap tm_q;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)d.D, (cuuint64_t)d.Hq, (cuuint64_t)d.M, (cuuint64_t)d.B};
    const cuuint64_t strides[3] = {(cuuint64_t)d.D * 2, (cuuint64_t)d.Hq * d.D * 2,
                                   (cuuint64_t)d.M * d.Hq * d.D * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)group, (cuuint32_t)d.M, 1};
    if (!make_map(&tm_q, a.q, dims, strides, box)) return cudaErrorInvalidValue;
  }

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int G = sms < kMaxAttnCtas ? sms : kMaxAttnCtas;

  {
    PdlLaunch L(dim3(d.B), dim3(kPrepThreads), 0, st);
    e = cudaLaunchKernelEx(&L.cfg, attn_prep_kernel, a.block_table, a.ctx_lens,
                           a.parent, d, G, ntiles, pre, rq, starts, pairs, anc, arrivals,
                           static_cast<__nv_bfloat16*>(a.out), a.lse, status);
    if (e != cudaSuccess) return e;
  }
  ++*launches;
  const bool wide = d.M > 64, short_wait = wait_limit_cycles(d) < ptx::kShortWait;
  auto kern = wide ? (short_wait ? attn_tc_kernel<true, true> : attn_tc_kernel<true, false>)
                   : (short_wait ? attn_tc_kernel<false, true> : attn_tc_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const float qscale2 = a.scale * 1.4426950408889634f;
  {
    PdlLaunch L(dim3(G), dim3(kThreads), kSmemBytes, st);
    e = cudaLaunchKernelEx(&L.cfg, kern, tm_q,
                           static_cast<const __nv_bfloat16*>(a.k_new),
                           static_cast<const __nv_bfloat16*>(a.v_new),
                           static_cast<__nv_bfloat16*>(a.k_cache),
                           static_cast<__nv_bfloat16*>(a.v_cache), a.block_table,
                           (const int4*)rq, (const int4*)starts,
                           a.parent != nullptr ? (const ulonglong2*)anc : nullptr, pairs, d,
                           qscale2, part, static_cast<__nv_bfloat16*>(a.out), a.lse, status);
    if (e != cudaSuccess) return e;
  }
  ++*launches;
  return cudaGetLastError();
}

}  // namespace specv
