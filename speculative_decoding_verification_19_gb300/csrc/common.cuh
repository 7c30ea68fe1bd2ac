// Shared device helpers of the verify-step kernels: element loads, status
// flags, warp reductions and the workspace layout.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

namespace specv {

constexpr int kBlock = 16;          // tokens per KV block
constexpr int kMaxNodes = 128;      // new rows (draft-tree nodes incl. the root) per request
constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Unpack the 8 bf16 (or 4 fp32) values of one 16-byte vector to fp32.
__device__ __forceinline__ void unpack16(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void unpack16(const uint4& v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

template <typename T> struct Vec16 { static constexpr int n = 16 / sizeof(T); };

// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32): relative
// error about 2^-22, results below 2^-126 flush to zero.  On sm_103 it is
// several times cheaper per element than exp2f(), which matters in the
// per-logit and per-score loops.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// status word (bit (1 << code) per raised spec_status code)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_status(uint32_t* status, int code) {
  atomicOr(status, 1u << code);
}
__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

// ---------------------------------------------------------------------------
// warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
  return __reduce_or_sync(0xffffffffu, (unsigned)v);
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with PdlLaunch may start
// while its predecessor on the stream drains; it must call pdl_wait() before
// touching memory a predecessor writes (which also keeps the chain
// transitive), and calls pdl_trigger() early to let its own dependents launch.
// Pointers to what a predecessor kernel of the chain writes are never
// __restrict__: a restrict-qualified load may be moved above pdl_wait (or
// served by the read-only path) and then see the memory before the write.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

struct PdlLaunch {  // use in place: cfg points at attr
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg;
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
  }
  PdlLaunch(const PdlLaunch&) = delete;
  PdlLaunch& operator=(const PdlLaunch&) = delete;
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// Every spin-wait of the kernels gives up after a limit of SM clocks and
// raises SPEC_ERR_TIMEOUT.  The caller may lower the limit
// (spec_dims.wait_limit_kcycles, in thousands of clocks); waits for work a
// CTA has already issued (copies into its shared memory, MMAs into its
// tensor memory) keep the default limit whatever the caller asks, because
// the CTA must not exit before that work lands.
constexpr uint64_t kDefaultWaitCycles = 4000000000ull;  // about 2 s at 2 GHz
__host__ __device__ __forceinline__ uint64_t wait_limit_cycles(const spec_dims& d) {
  return d.wait_limit_kcycles > 0 ? (uint64_t)d.wait_limit_kcycles * 1000ull : kDefaultWaitCycles;
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// workspace layout (computed identically by every entry point)
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t status_off;      // uint32 status word
  size_t attn_ok_off;     // [B] int32 per-request verdict of the append
  size_t tc_ntiles_off;   // [B] int32 64-key tiles per (request, head)
  size_t tc_pre_off;      // [2][B+1] int64 prefixes of tiles and of split costs over requests
  size_t tc_rq_off;       // [B] int4 per request: ctx, tiles per head, next request with tiles
  size_t tc_start_off;    // [kMaxAttnCtas+1][2] int4 per CTA: first tile, its (request, head,
                          // tile), the request's record and the end tile
  size_t tc_pair_off;     // [B*Hkv] int32 per (request, KV head): tiles run by the later CTAs
  size_t tc_anc_off;      // [B*M] 128-bit ancestor-or-self mask of every tree row (2 u64)
  size_t tc_sync_off;     // uint32 arrival count of the request-check kernel
  size_t attn_off;        // split-KV partials of either attention path (f32)
  size_t attn_bytes;
  int split_keys;         // keys per split (multiple of 16)
  int max_splits;
  int rows;               // R = group * M
  size_t rs_off;          // reject-sample chunk stats: [B, 2, M, n_chunks] RowStat
  size_t rs_bytes;
  size_t rs_draw_off;     // [B] DrawState: residual draws left for pass 3
  size_t rs_zsum_off;     // [B, n_chunks] f64: residual mass of each statistics chunk
  size_t rs_filt_off;     // [B, 2, M] 16-byte kept prefix of each filtered row
  size_t rs_tail_off;     // [B] u32 slices of the chain tail kernel finished per request
  size_t lm_part_off;     // LM heads' split statistics: [2][units][4][128] RowStat
  size_t lm_cnt_off;      // [2][units][4] u32 pieces finished per (unit, 32-row warp)
  int64_t lm_units;       // units laid out (0: LM-head units are not split)
  int rs_chunk;           // logits per statistics chunk
  int rs_chunks;          // statistics chunks per row
  // the one-kernel reject path (laid out by rsf_layout)
  size_t rsf_ctl_off;     // 64 u32 control words
  size_t rsf_norm_off;    // [B, 2M] 16-byte row normalisers
  size_t rsf_rowcnt_off;  // [B, 2M] u32 statistics chunks finished per row
  size_t rsf_req_off;     // [B] u32 rows finished per request
  size_t rsf_list_off;    // [B] 48-byte residual entries in the order posted
  size_t rsf_rescnt_off;  // [B] u32 residual units finished per request
  size_t total;
};

WsLayout workspace_layout(const spec_dims& d);

// Checks of the dims every entry point shares (counts, M, block size,
// dtypes, the wait limit and the kernel selectors).
spec_status check_common(const spec_dims* d);

}  // namespace specv
