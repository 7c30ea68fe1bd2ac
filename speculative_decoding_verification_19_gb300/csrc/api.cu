// C ABI of the verify step: argument checks, workspace layout and launches.
// Every check that the host can make happens here, before anything is
// enqueued; the kernels only check what lives in device memory.
#include <math.h>
#include <string.h>

#include "attn.cuh"
#include "common.cuh"
#include "kv_commit.cuh"
#include "philox.cuh"
#include "lm_head.cuh"
#include "reject_sample.cuh"

namespace specv {

static thread_local int32_t g_launches = 0;

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int attn_split_keys(const spec_dims& d) {
  // Aim for about eight CTAs per SM over the whole batch (152 SMs), with
  // ranges of 256..4096 keys in whole 32-key tiles.
  const int64_t max_keys = (int64_t)d.max_blocks * kBlock;
  int64_t s = (int64_t)d.B * d.Hkv * max_keys / 1216;
  s = (s + 31) / 32 * 32;
  if (s < 256) s = 256;
  if (s > 4096) s = 4096;
  return (int)s;
}

WsLayout workspace_layout(const spec_dims& d) {
  WsLayout L;
  memset(&L, 0, sizeof(L));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status_off = take(16);
  L.attn_ok_off = take(sizeof(int32_t) * (size_t)d.B);
  L.tc_ntiles_off = take(sizeof(int32_t) * (size_t)d.B);
  L.tc_pre_off = take(sizeof(int64_t) * 2 * ((size_t)d.B + 1));
  L.tc_rq_off = take(16 * (size_t)d.B);
  L.tc_start_off = take(32 * ((size_t)kMaxAttnCtas + 1));
  L.tc_pair_off = take(sizeof(int32_t) * (size_t)d.B * (size_t)(d.Hkv > 0 ? d.Hkv : 0));
  L.tc_anc_off = take(2 * sizeof(uint64_t) * (size_t)d.B * d.M);
  L.tc_sync_off = take(16);
  const int group = d.Hkv > 0 ? d.Hq / d.Hkv : 0;
  L.rows = group * d.M;
  L.split_keys = attn_split_keys(d);
  L.max_splits = (int)ceil_div64((int64_t)d.max_blocks * kBlock, L.split_keys);
  L.attn_bytes = sizeof(float) * (size_t)d.B * d.Hkv * L.max_splits * L.rows * (d.D + 1);
  const size_t tc_bytes = d.Hkv > 0 ? sizeof(float) * attn_tc_part_floats(d) : 0;
  if (tc_bytes > L.attn_bytes) L.attn_bytes = tc_bytes;
  L.attn_off = take(L.attn_bytes);
  L.rs_chunk = rs_chunk_elems(d.logits_dtype);
  L.rs_chunks = (int)ceil_div64(d.V, L.rs_chunk);
  L.rs_bytes = sizeof(RowStat) * (size_t)d.B * 2 * d.M * L.rs_chunks;
  L.rs_off = take(L.rs_bytes);
  L.rs_draw_off = take(sizeof(DrawState) * (size_t)d.B);
  L.rs_zsum_off = take(sizeof(double) * (size_t)d.B * L.rs_chunks);
  L.rs_filt_off = take(sizeof(FilterInfo) * (size_t)d.B * 2 * d.M);
  // the chain tail: per request, slices finished, then residual chunks
  // claimed; then the statistics stream's pool counters (claimed, warps done)
  L.rs_tail_off = take(sizeof(uint32_t) * (2 * (size_t)d.B + 2));
  // the LM heads' split statistics (rows B * M, bf16 logits)
  const int64_t lm_units = (int64_t)ceil_div64((int64_t)d.B * d.M, 128) * L.rs_chunks;
  if (d.logits_dtype == SPEC_BF16 && lm_units <= kLmSplitMaxUnits) {
    L.lm_units = lm_units;
    L.lm_part_off = take(sizeof(RowStat) * 2 * (size_t)lm_units * kLmMaxPieces * 128);
    L.lm_cnt_off = take(sizeof(uint32_t) * 2 * (size_t)lm_units * 4);
  }
  off = rsf_layout(d, off, &L);
  L.total = off;
  return L;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

spec_status check_common(const spec_dims* d) {
  if (d == nullptr) return SPEC_ERR_INVALID_ARG;
  if (d->B < 1 || d->M < 1) return SPEC_ERR_INVALID_ARG;
  if (d->M > kMaxNodes) return SPEC_ERR_UNSUPPORTED;
  if (d->block != kBlock) return SPEC_ERR_UNSUPPORTED;
  if ((d->kv_dtype != SPEC_BF16 && d->kv_dtype != SPEC_F32) ||
      (d->logits_dtype != SPEC_BF16 && d->logits_dtype != SPEC_F32))
    return SPEC_ERR_INVALID_ARG;
  if (d->wait_limit_kcycles < 0) return SPEC_ERR_INVALID_ARG;
  if (d->reject_impl < SPEC_REJECT_AUTO || d->reject_impl > SPEC_REJECT_FUSED)
    return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

static spec_status check_kv(const spec_dims* d) {
  if (d->B > 65535) return SPEC_ERR_UNSUPPORTED;  // grid y/z limit of the attention launch
  if (d->Hq < 1 || d->Hkv < 1 || d->Hq % d->Hkv != 0) return SPEC_ERR_INVALID_ARG;
  if (d->D != 64 && d->D != 128) return SPEC_ERR_UNSUPPORTED;
  if (d->max_blocks < 1 || d->num_blocks < 1) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

static spec_status check_ws(const spec_dims* d, void* ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned16(ws)) return SPEC_ERR_INVALID_ARG;
  if (ws_bytes < workspace_layout(*d).total) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

static spec_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

}  // namespace specv

using namespace specv;

extern "C" {

size_t spec_workspace_size(const spec_dims* dims) {
  if (check_common(dims) != SPEC_OK) return 0;
  return workspace_layout(*dims).total;
}

spec_status spec_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes == 0) return SPEC_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

spec_status spec_get_device_status(void* ws, void* stream, int32_t* flags, int32_t clear) {
  if (ws == nullptr || flags == nullptr) return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  *flags = (int32_t)v;
  if (clear) {
    e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

spec_status spec_verify_attn(const void* q, const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, const int32_t* block_table, const int32_t* ctx_lens,
                             const int32_t* parent, void* out, float* lse, const spec_dims* dims,
                             void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  spec_status s = check_common(dims);
  if (s != SPEC_OK) return s;
  if ((s = check_kv(dims)) != SPEC_OK) return s;
  if ((s = check_ws(dims, ws, ws_bytes)) != SPEC_OK) return s;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_table || !ctx_lens || !out)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out))
    return SPEC_ERR_INVALID_ARG;
  const int R = (dims->Hq / dims->Hkv) * dims->M;
  // kernel choice: the tensor-core kernel whenever it supports the shape
  // (bf16, D = 128, up to 128 rows per KV head): even a few rows per KV head
  // run faster there than on CUDA cores; CUDA cores otherwise
  const bool tc_ok = dims->kv_dtype == SPEC_BF16 && dims->D == 128 && R <= 128 &&
                     (int64_t)dims->B * dims->Hkv *
                             ceil_div64((int64_t)dims->max_blocks * kBlock, 64) <
                         ((int64_t)1 << 31);
  const bool simt_ok = R <= 128;
  bool use_tc;
  if (dims->attn_impl == SPEC_ATTN_TENSOR_CORES) {
    if (!tc_ok) return SPEC_ERR_UNSUPPORTED;
    use_tc = true;
  } else if (dims->attn_impl == SPEC_ATTN_CUDA_CORES) {
    if (!simt_ok) return SPEC_ERR_UNSUPPORTED;
    use_tc = false;
  } else if (dims->attn_impl == SPEC_ATTN_AUTO) {
    use_tc = tc_ok;
    if (!use_tc && !simt_ok) return SPEC_ERR_UNSUPPORTED;
  } else {
    return SPEC_ERR_INVALID_ARG;
  }
  const WsLayout lay = workspace_layout(*dims);
  AttnArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.parent = parent;
  a.out = out;
  a.lse = lse;
  a.d = *dims;
  a.scale = dims->softmax_scale != 0.f ? dims->softmax_scale : 1.0f / sqrtf((float)dims->D);
  a.ws = ws;
  int launches = 0;
  const cudaError_t e = use_tc ? attn_launch_tc(a, lay, static_cast<cudaStream_t>(stream), &launches)
                               : attn_launch_simt(a, lay, static_cast<cudaStream_t>(stream), &launches);
  g_launches = launches;
  return from_cuda(e);
}

static spec_status reject_common(const void* target_logits, const void* draft_logits,
                                 const int32_t* tokens, const int32_t* parent,
                                 const float* temperature, const int32_t* top_k,
                                 const float* top_p, uint64_t seed, uint64_t offset,
                                 uint64_t b_base, int32_t* out_tokens, int32_t* path,
                                 int32_t* accepted_len, float* probe, const spec_dims* dims,
                                 void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  spec_status s = check_common(dims);
  if (s != SPEC_OK) return s;
  if ((s = check_ws(dims, ws, ws_bytes)) != SPEC_OK) return s;
  if (dims->V < 1) return SPEC_ERR_INVALID_ARG;
  if (dims->V > rs_max_vocab(dims->logits_dtype)) return SPEC_ERR_UNSUPPORTED;
  {
    const WsLayout l = workspace_layout(*dims);
    if ((int64_t)l.rs_chunks * 2 * dims->M * dims->B >= (int64_t)1 << 31) return SPEC_ERR_UNSUPPORTED;
  }
  if (!target_logits || !draft_logits || !tokens || !temperature || !out_tokens || !path ||
      !accepted_len)
    return SPEC_ERR_INVALID_ARG;
  if ((top_k != nullptr || top_p != nullptr) && dims->reject_impl == SPEC_REJECT_FUSED)
    return SPEC_ERR_UNSUPPORTED;  // the one-kernel path has no filters
  const WsLayout lay = workspace_layout(*dims);
  RsArgs a;
  a.target = target_logits;
  a.draft = draft_logits;
  a.tokens = tokens;
  a.parent = parent;
  a.temperature = temperature;
  a.top_k = top_k;
  a.top_p = top_p;
  a.seed = seed;
  a.offset = offset;
  a.b_base = b_base;
  a.out_tokens = out_tokens;
  a.path = path;
  a.accepted_len = accepted_len;
  a.probe = probe;
  a.d = *dims;
  a.ws = ws;
  int launches = 0;
  const cudaError_t e = rs_launch(a, lay, static_cast<cudaStream_t>(stream), &launches);
  g_launches = launches;
  if (e == cudaErrorNotSupported) return SPEC_ERR_UNSUPPORTED;
  return from_cuda(e);
}

spec_status spec_reject_sample(const void* target_logits, const void* draft_logits,
                               const int32_t* tokens, const int32_t* parent,
                               const float* temperature, uint64_t seed, uint64_t offset,
                               uint64_t b_base, int32_t* out_tokens, int32_t* path,
                               int32_t* accepted_len, float* probe, const spec_dims* dims,
                               void* ws, size_t ws_bytes, void* stream) {
  return reject_common(target_logits, draft_logits, tokens, parent, temperature, nullptr,
                       nullptr, seed, offset, b_base, out_tokens, path, accepted_len, probe, dims,
                       ws, ws_bytes, stream);
}

spec_status spec_reject_sample_filtered(const void* target_logits, const void* draft_logits,
                                        const int32_t* tokens, const int32_t* parent,
                                        const float* temperature, const int32_t* top_k,
                                        const float* top_p, uint64_t seed, uint64_t offset,
                                        uint64_t b_base, int32_t* out_tokens, int32_t* path,
                                        int32_t* accepted_len, float* probe,
                                        const spec_dims* dims, void* ws, size_t ws_bytes,
                                        void* stream) {
  return reject_common(target_logits, draft_logits, tokens, parent, temperature, top_k, top_p,
                       seed, offset, b_base, out_tokens, path, accepted_len, probe, dims, ws,
                       ws_bytes, stream);
}

spec_status spec_lm_head(const void* hidden, const void* weight, int32_t rows, int32_t H,
                         int32_t V, void* logits, void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  if (!hidden || !weight || !logits || ws == nullptr || ws_bytes < 16 || !aligned16(ws))
    return SPEC_ERR_INVALID_ARG;
  if (rows < 1 || H < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!lm_head_supported(rows, H, V)) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(logits)) return SPEC_ERR_INVALID_ARG;
  spec_dims d;
  memset(&d, 0, sizeof(d));  // the default wait limit
  int launches = 0;
  const cudaError_t e =
      lm_head_launch(hidden, weight, rows, H, V, logits, nullptr, 0, 1, 0, nullptr, d,
                     static_cast<uint32_t*>(ws), nullptr, nullptr,
                     static_cast<cudaStream_t>(stream), &launches);
  g_launches = launches;
  return e == cudaErrorInvalidValue ? SPEC_ERR_UNSUPPORTED : from_cuda(e);
}

spec_status spec_reject_sample_lm_head(const void* hidden_target, const void* weight_target,
                                       int32_t Ht, const void* hidden_draft,
                                       const void* weight_draft, int32_t Hd, void* target_logits,
                                       void* draft_logits, const int32_t* tokens,
                                       const int32_t* parent, const float* temperature,
                                       uint64_t seed, uint64_t offset, uint64_t b_base,
                                       int32_t* out_tokens, int32_t* path, int32_t* accepted_len,
                                       float* probe, const spec_dims* dims, void* ws,
                                       size_t ws_bytes, void* stream) {
  g_launches = 0;
  spec_status s = check_common(dims);
  if (s != SPEC_OK) return s;
  if ((s = check_ws(dims, ws, ws_bytes)) != SPEC_OK) return s;
  if (!hidden_target || !weight_target || !hidden_draft || !weight_draft || !target_logits ||
      !draft_logits || !tokens || !temperature || !out_tokens || !path || !accepted_len)
    return SPEC_ERR_INVALID_ARG;
  if (dims->logits_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (dims->reject_impl == SPEC_REJECT_FUSED) return SPEC_ERR_UNSUPPORTED;
  const int R = dims->B * dims->M;
  if ((int64_t)dims->B * dims->M >= ((int64_t)1 << 31) / 2) return SPEC_ERR_UNSUPPORTED;
  if (!lm_head_supported(R, Ht, dims->V) || !lm_head_supported(R, Hd, dims->V))
    return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(hidden_target) || !aligned16(weight_target) || !aligned16(hidden_draft) ||
      !aligned16(weight_draft) || !aligned16(target_logits) || !aligned16(draft_logits))
    return SPEC_ERR_INVALID_ARG;
  const WsLayout lay = workspace_layout(*dims);
  if ((int64_t)lay.rs_chunks * 2 * dims->M * dims->B >= (int64_t)1 << 31) return SPEC_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  RowStat* stats = reinterpret_cast<RowStat*>(w + lay.rs_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(w + lay.status_off);
  int launches = 0;
  // the split statistics' workspace, when laid out for these rows
  const bool split = lay.lm_units > 0 && lay.lm_units == lm_head_units(R, dims->V);
  RowStat* part = split ? reinterpret_cast<RowStat*>(w + lay.lm_part_off) : nullptr;
  uint32_t* cnt = split ? reinterpret_cast<uint32_t*>(w + lay.lm_cnt_off) : nullptr;
  cudaError_t e = lm_head_launch(hidden_target, weight_target, R, Ht, dims->V, target_logits,
                                 stats, 0, dims->M, lay.rs_chunks, temperature, *dims, status,
                                 part, cnt, st, &launches);
  if (e == cudaSuccess)
    e = lm_head_launch(hidden_draft, weight_draft, R, Hd, dims->V, draft_logits, stats, 1,
                       dims->M, lay.rs_chunks, temperature, *dims, status, part, cnt, st,
                       &launches);
  if (e != cudaSuccess) {
    g_launches = launches;
    return e == cudaErrorInvalidValue ? SPEC_ERR_UNSUPPORTED : SPEC_ERR_CUDA;
  }
  RsArgs a;
  a.target = target_logits;
  a.draft = draft_logits;
  a.tokens = tokens;
  a.parent = parent;
  a.temperature = temperature;
  a.top_k = nullptr;
  a.top_p = nullptr;
  a.seed = seed;
  a.offset = offset;
  a.b_base = b_base;
  a.out_tokens = out_tokens;
  a.path = path;
  a.accepted_len = accepted_len;
  a.probe = probe;
  a.d = *dims;
  a.d.reject_impl = SPEC_REJECT_STAGED;
  a.ws = ws;
  a.stats_ready = true;
  e = rs_launch(a, lay, st, &launches);
  g_launches = launches;
  return from_cuda(e);
}

spec_status kv_commit(void* k_cache, void* v_cache, const int32_t* block_table,
                      const int32_t* ctx_lens, int32_t* new_ctx_lens, const int32_t* path,
                      const int32_t* accepted_len, const spec_dims* dims, void* ws,
                      size_t ws_bytes, void* stream) {
  g_launches = 0;
  spec_status s = check_common(dims);
  if (s != SPEC_OK) return s;
  if ((s = check_kv(dims)) != SPEC_OK) return s;
  if ((s = check_ws(dims, ws, ws_bytes)) != SPEC_OK) return s;
  if (!k_cache || !v_cache || !block_table || !ctx_lens || !new_ctx_lens || !path || !accepted_len)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return SPEC_ERR_INVALID_ARG;
  const WsLayout lay = workspace_layout(*dims);
  CommitArgs a;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.new_ctx_lens = new_ctx_lens;
  a.path = path;
  a.accepted_len = accepted_len;
  a.d = *dims;
  a.ws = ws;
  int launches = 0;
  const cudaError_t e = commit_launch(a, lay, static_cast<cudaStream_t>(stream), &launches);
  g_launches = launches;
  return from_cuda(e);
}

void spec_philox_block(const uint64_t key[2], const uint64_t counter[4], uint64_t out[4]) {
  const Philox4 r = philox4x64_10(counter[0], counter[1], counter[2], counter[3], key[0], key[1]);
  for (int i = 0; i < 4; ++i) out[i] = r.w[i];
}

const char* spec_status_string(int32_t status) {
  switch (status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_CAPACITY: return "SPEC_ERR_CAPACITY";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_NONFINITE: return "SPEC_ERR_NONFINITE";
    case SPEC_ERR_DEVICE_BOUNDS: return "SPEC_ERR_DEVICE_BOUNDS";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    default: return "SPEC_ERR_UNKNOWN";
  }
}

int32_t spec_last_launch_count(void) { return g_launches; }

}  // extern "C"
