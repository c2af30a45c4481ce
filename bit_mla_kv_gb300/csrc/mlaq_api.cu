// C-ABI entry points of libmlaq: argument checking and kernel launches.
#include <stdlib.h>
#include <string.h>

#include "mlaq_internal.cuh"

namespace mlaq {
size_t workspace_bytes_for(int max_seqs, int max_heads);
int launch_decode_static(int mode, const void* codes, const void* meta, const void* ring, int num_pages,
                         int max_pages_per_seq, const uint16_t* q_latent, const uint16_t* q_rope,
                         const int32_t* page_table, const int32_t* seq_lens, int B, int H, float scale,
                         uint16_t* out, float* lse, int32_t* dev_status, cudaStream_t s);
}

namespace mlaq {
// One warp waits on an mbarrier that nothing (arrive = 0) or its own thread 0
// (arrive = 1) completes, through the bounded wait of the decode kernel.
__global__ void wait_probe_kernel(int32_t* status, uint64_t limit_ns, int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (arrive) mbar_arrive_expect_tx(&bar, 0);
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
  if (threadIdx.x == 0) *status = ok ? 0 : MLAQ_DEV_TIMEOUT;
}
}  // namespace mlaq

using namespace mlaq;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool valid_mode(int m) { return m == MLAQ_C4R4 || m == MLAQ_C2R4 || m == MLAQ_BF16; }

extern "C" {

const char* mlaq_status_string(int status) {
  switch (status) {
    case MLAQ_OK: return "ok";
    case MLAQ_ERR_NULL: return "required pointer is NULL";
    case MLAQ_ERR_MODE: return "unknown cache mode";
    case MLAQ_ERR_SHAPE: return "size outside the supported range";
    case MLAQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MLAQ_ERR_CAPACITY: return "batch or heads exceed the cache capacity";
    case MLAQ_ERR_CUDA: return "CUDA runtime error";
    case MLAQ_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int mlaq_buffer_sizes(int mode, int32_t num_pages, int32_t max_seqs, int32_t max_heads, size_t* codes_bytes,
                      size_t* meta_bytes, size_t* ring_bytes, size_t* workspace_bytes) {
  if (!valid_mode(mode)) return MLAQ_ERR_MODE;
  if (!codes_bytes || !meta_bytes || !ring_bytes || !workspace_bytes) return MLAQ_ERR_NULL;
  if (num_pages <= 0 || max_seqs <= 0 || max_seqs > kMaxSeqs || max_heads < 16 || max_heads > 128 || max_heads % 16)
    return MLAQ_ERR_SHAPE;
  *codes_bytes = (size_t)num_pages * page_code_bytes(mode);
  *meta_bytes = mode == MLAQ_BF16 ? 0 : (size_t)num_pages * kMetaPage;
  *ring_bytes = mode == MLAQ_BF16 ? 0 : (size_t)max_seqs * kRing * kD * 2;
  *workspace_bytes = workspace_bytes_for(max_seqs, max_heads);
  return MLAQ_OK;
}

int mlaq_cache_create(mlaq_cache** out, int mode, int32_t num_pages, int32_t max_seqs, int32_t max_pages_per_seq,
                      int32_t max_heads, void* codes, void* meta, void* ring, void* workspace,
                      size_t workspace_bytes) {
  if (!out) return MLAQ_ERR_NULL;
  *out = nullptr;
  if (!valid_mode(mode)) return MLAQ_ERR_MODE;
  if (num_pages <= 0 || max_seqs <= 0 || max_seqs > kMaxSeqs || max_pages_per_seq <= 0 || max_heads < 16 ||
      max_heads > 128 || max_heads % 16 || !plan_cost_fits(max_seqs, max_pages_per_seq))
    return MLAQ_ERR_SHAPE;
  if (!codes || !workspace || (mode != MLAQ_BF16 && (!meta || !ring))) return MLAQ_ERR_NULL;
  if (!aligned16(codes) || !aligned16(workspace) || (mode != MLAQ_BF16 && (!aligned16(meta) || !aligned16(ring))))
    return MLAQ_ERR_ALIGN;
  if (workspace_bytes < workspace_bytes_for(max_seqs, max_heads)) return MLAQ_ERR_WORKSPACE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLAQ_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLAQ_ERR_CUDA;
  mlaq_cache* c = static_cast<mlaq_cache*>(calloc(1, sizeof(mlaq_cache)));
  if (!c) return MLAQ_ERR_NULL;
  c->mode = mode;
  c->num_pages = num_pages;
  c->max_seqs = max_seqs;
  c->max_pages_per_seq = max_pages_per_seq;
  c->max_heads = max_heads;
  c->codes = codes;
  c->meta = meta;
  c->ring = ring;
  c->workspace = workspace;
  c->workspace_bytes = workspace_bytes;
  c->num_sms = sms;
  c->decode_ctas = 0;  // the kernel's own default (one wave) until mlaq_set_decode_ctas
  c->cost_step = kDefCostStep;
  c->cost_ring = kDefCostRing;
  c->cost_item = kDefCostItem;
  *out = c;
  return MLAQ_OK;
}

int mlaq_cache_destroy(mlaq_cache* c) {
  if (!c) return MLAQ_ERR_NULL;
  if (c->timing_events) {
    cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(c->timing_events);
    for (int k = 0; k < 2 * c->timing_max; ++k) cudaEventDestroy(ev[k]);
    free(c->timing_events);
  }
  free(c);
  return MLAQ_OK;
}

int mlaq_append(mlaq_cache* c, const int32_t* page_table, int32_t* seq_lens, int32_t B, const uint16_t* c_latent,
                const uint16_t* k_rope, int32_t n_new, const int32_t* cu_new, int32_t total_new,
                struct CUstream_st* stream) {
  if (!c || !page_table || !seq_lens) return MLAQ_ERR_NULL;
  if (B <= 0) return MLAQ_ERR_SHAPE;
  if (B > c->max_seqs) return MLAQ_ERR_CAPACITY;
  if (cu_new == nullptr) {
    if (n_new < 0) return MLAQ_ERR_SHAPE;
    if ((int64_t)B * n_new > (int64_t)0x7fffffff) return MLAQ_ERR_SHAPE;
    total_new = B * n_new;
  } else if (total_new < 0) {
    return MLAQ_ERR_SHAPE;
  }
  if (total_new > 0 && (!c_latent || !k_rope)) return MLAQ_ERR_NULL;
  if (total_new > 0 && (!aligned16(c_latent) || !aligned16(k_rope))) return MLAQ_ERR_ALIGN;
  cudaError_t e = launch_append(c, page_table, seq_lens, B, c_latent, k_rope, n_new, cu_new, total_new,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLAQ_OK : MLAQ_ERR_CUDA;
}

int mlaq_decode(mlaq_cache* c, const uint16_t* q_latent, const uint16_t* q_rope, const int32_t* page_table,
                const int32_t* seq_lens, int32_t B, int32_t H, float softmax_scale, uint16_t* out_latent,
                float* lse, struct CUstream_st* stream) {
  if (!c || !q_latent || !q_rope || !page_table || !seq_lens || !out_latent || !lse) return MLAQ_ERR_NULL;
  if (B <= 0 || H < 16 || H > 128 || H % 16) return MLAQ_ERR_SHAPE;
  if (B > c->max_seqs || H > c->max_heads) return MLAQ_ERR_CAPACITY;
  if (!aligned16(q_latent) || !aligned16(q_rope) || !aligned16(out_latent)) return MLAQ_ERR_ALIGN;
  cudaError_t e = launch_decode(c, q_latent, q_rope, page_table, seq_lens, B, H, softmax_scale, out_latent, lse,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLAQ_OK : MLAQ_ERR_CUDA;
}

int mlaq_decode_mtp(mlaq_cache* c, const uint16_t* q_latent, const uint16_t* q_rope, const int32_t* page_table,
                    const int32_t* seq_lens, int32_t B, int32_t Q, int32_t H, float softmax_scale,
                    uint16_t* out_latent, float* lse, struct CUstream_st* stream) {
  if (!c || !q_latent || !q_rope || !page_table || !seq_lens || !out_latent || !lse) return MLAQ_ERR_NULL;
  if (B <= 0 || Q <= 0 || H < 16 || H % 16 || Q * H > 128) return MLAQ_ERR_SHAPE;
  if (B > c->max_seqs || Q * H > c->max_heads) return MLAQ_ERR_CAPACITY;
  if (!aligned16(q_latent) || !aligned16(q_rope) || !aligned16(out_latent)) return MLAQ_ERR_ALIGN;
  // the Q query rows of a sequence are laid out as Q * H heads
  cudaError_t e = launch_decode(c, q_latent, q_rope, page_table, seq_lens, B, Q * H, softmax_scale, out_latent, lse,
                                reinterpret_cast<cudaStream_t>(stream), Q);
  return e == cudaSuccess ? MLAQ_OK : MLAQ_ERR_CUDA;
}

int mlaq_decode_noalloc(int mode, const void* codes, const void* meta, const void* ring, int32_t num_pages,
                        int32_t max_pages_per_seq, const uint16_t* q_latent, const uint16_t* q_rope,
                        const int32_t* page_table, const int32_t* seq_lens, int32_t B, int32_t H,
                        float softmax_scale, uint16_t* out_latent, float* lse, int32_t* dev_status,
                        struct CUstream_st* stream) {
  if (!valid_mode(mode)) return MLAQ_ERR_MODE;
  if (!codes || !q_latent || !q_rope || !page_table || !seq_lens || !out_latent || !lse) return MLAQ_ERR_NULL;
  if (mode != MLAQ_BF16 && (!meta || !ring)) return MLAQ_ERR_NULL;
  if (num_pages <= 0 || max_pages_per_seq <= 0) return MLAQ_ERR_SHAPE;
  if (B <= 0 || !plan_cost_fits(B, max_pages_per_seq)) return MLAQ_ERR_SHAPE;
  if (B <= 0 || B > kMaxSeqs || H < 16 || H > 128 || H % 16) return MLAQ_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(q_latent) || !aligned16(q_rope) || !aligned16(out_latent) ||
      (mode != MLAQ_BF16 && (!aligned16(meta) || !aligned16(ring))))
    return MLAQ_ERR_ALIGN;
  return launch_decode_static(mode, codes, meta, ring, num_pages, max_pages_per_seq, q_latent, q_rope, page_table,
                              seq_lens, B, H, softmax_scale, out_latent, lse, dev_status,
                              reinterpret_cast<cudaStream_t>(stream));
}

int mlaq_export_tokens(mlaq_cache* c, const int32_t* page_table, int32_t B, const int32_t* token_b,
                       const int32_t* token_t, int32_t n, uint8_t* codes_out, uint16_t* meta_out,
                       struct CUstream_st* stream) {
  if (!c || !page_table || !token_b || !token_t || !codes_out || !meta_out) return MLAQ_ERR_NULL;
  if (c->mode == MLAQ_BF16) return MLAQ_ERR_MODE;
  if (n < 0 || B <= 0) return MLAQ_ERR_SHAPE;
  cudaError_t e = launch_export(c, page_table, B, token_b, token_t, n, codes_out, meta_out,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLAQ_OK : MLAQ_ERR_CUDA;
}

int mlaq_cache_bytes(const mlaq_cache* c, const int32_t* seq_lens_host, int32_t B, size_t* policy_bytes,
                     size_t* bf16_bytes) {
  if (!c || !seq_lens_host || !policy_bytes || !bf16_bytes) return MLAQ_ERR_NULL;
  if (B < 0) return MLAQ_ERR_SHAPE;
  size_t pol = 0, ref = 0;
  const size_t tok_packed = (size_t)token_bytes(c->mode) + (c->mode == MLAQ_BF16 ? 0 : kMetaTok);
  for (int b = 0; b < B; ++b) {
    const size_t L = seq_lens_host[b] > 0 ? (size_t)seq_lens_host[b] : 0;
    const size_t pages = (L + kPage - 1) / kPage;
    const size_t map = pages * sizeof(int32_t);
    pol += pages * kPage * tok_packed + map + (c->mode == MLAQ_BF16 ? 0 : (size_t)kRing * kD * 2);
    ref += pages * kPage * kD * 2 + map;
  }
  *policy_bytes = pol;
  *bf16_bytes = ref;
  return MLAQ_OK;
}

int mlaq_get_device_status(mlaq_cache* c, struct CUstream_st* stream, int32_t* status) {
  if (!c || !status) return MLAQ_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLAQ_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, static_cast<char*>(c->workspace) + kWsStatus, sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return MLAQ_ERR_CUDA;
  *status = v;
  return MLAQ_OK;
}

int mlaq_clear_device_status(mlaq_cache* c, struct CUstream_st* stream) {
  if (!c) return MLAQ_ERR_NULL;
  if (cudaMemsetAsync(static_cast<char*>(c->workspace) + kWsStatus, 0, sizeof(int),
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLAQ_ERR_CUDA;
  return MLAQ_OK;
}

int mlaq_timing_enable(mlaq_cache* c, int32_t max_calls) {
  if (!c) return MLAQ_ERR_NULL;
  if (max_calls < 0) return MLAQ_ERR_SHAPE;
  if (c->timing_events) {
    cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(c->timing_events);
    for (int k = 0; k < 2 * c->timing_max; ++k) cudaEventDestroy(ev[k]);
    free(c->timing_events);
    c->timing_events = nullptr;
    c->timing_max = 0;
    c->timing_n = 0;
  }
  if (max_calls == 0) return MLAQ_OK;  // timing off
  cudaEvent_t* ev = static_cast<cudaEvent_t*>(calloc(2 * (size_t)max_calls, sizeof(cudaEvent_t)));
  if (!ev) return MLAQ_ERR_NULL;
  for (int k = 0; k < 2 * max_calls; ++k)
    if (cudaEventCreate(&ev[k]) != cudaSuccess) {
      for (int j = 0; j < k; ++j) cudaEventDestroy(ev[j]);
      free(ev);
      return MLAQ_ERR_CUDA;
    }
  c->timing_events = reinterpret_cast<void**>(ev);
  c->timing_max = max_calls;
  c->timing_n = 0;
  return MLAQ_OK;
}

int mlaq_timing_read(mlaq_cache* c, float* ms_out, int32_t* n) {
  if (!c || !ms_out || !n) return MLAQ_ERR_NULL;
  if (!c->timing_events) {
    *n = 0;
    return MLAQ_OK;
  }
  cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(c->timing_events);
  for (int k = 0; k < c->timing_n; ++k) {
    if (cudaEventSynchronize(ev[2 * k + 1]) != cudaSuccess) return MLAQ_ERR_CUDA;
    if (cudaEventElapsedTime(&ms_out[k], ev[2 * k], ev[2 * k + 1]) != cudaSuccess) return MLAQ_ERR_CUDA;
  }
  *n = c->timing_n;
  c->timing_n = 0;
  return MLAQ_OK;
}

int mlaq_set_decode_ctas(mlaq_cache* c, int32_t ctas) {
  if (!c) return MLAQ_ERR_NULL;
  if (ctas <= 0 || ctas > kMaxPlanCtas) return MLAQ_ERR_SHAPE;
  c->decode_ctas = ctas;
  c->decode_ctas_set = 1;
  return MLAQ_OK;
}

int mlaq_set_decode_variant(mlaq_cache* c, int32_t variant) {
  if (!c) return MLAQ_ERR_NULL;
  if (variant < 0 || variant > 2) return MLAQ_ERR_SHAPE;
  c->decode_variant = variant;
  return MLAQ_OK;
}

int mlaq_set_plan_costs(mlaq_cache* c, int32_t step, int32_t ring, int32_t item) {
  if (!c) return MLAQ_ERR_NULL;
  if (step < 1 || 4 * step > kPlanCostPerPage || ring < 1 || item < 0 ||
      item + ring * ((kRing + 15) / 16) > kPlanCostRingMax)  // 9 ring chunks of 16 slots
    return MLAQ_ERR_SHAPE;
  c->cost_step = step;
  c->cost_ring = ring;
  c->cost_item = item;
  return MLAQ_OK;
}

int mlaq_debug_wait_probe(int32_t* status, int32_t wait_us, int32_t arrive, struct CUstream_st* stream) {
  if (!status) return MLAQ_ERR_NULL;
  if (wait_us < 1 || wait_us > 100000 || (arrive != 0 && arrive != 1)) return MLAQ_ERR_SHAPE;
  wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, (uint64_t)wait_us * 1000u, arrive);
  return cudaGetLastError() == cudaSuccess ? MLAQ_OK : MLAQ_ERR_CUDA;
}

}  // extern "C"
