// C ABI of libcosa (declared in include/cosa.h): host-side argument checks, TMA tensor-map
// encoding, and the launches of the KAP and OSK kernels.  No allocation, no host copies.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "cosa.h"
#include "internal.h"

namespace {

using cosa::KapLaunch;
using cosa::OskLaunch;

constexpr int kMaxQueryBlocksKap = 4096;
constexpr int kMaxQueryBlocksOsk = 32768;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Checks shared by both calls.  Returns COSA_OK or an error code.
int check_common(const cosa_params* p) {
  if (p == nullptr) return COSA_ERR_INVALID_ARG;
  if (p->num_reqs < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1) return COSA_ERR_INVALID_ARG;
  if (p->num_q_heads % p->num_kv_heads != 0) return COSA_ERR_INVALID_ARG;
  if (p->total_tokens < 0 || p->max_seqlen < 1 || p->num_pages < 1 || p->max_pages_per_req < 1) return COSA_ERR_INVALID_ARG;
  if (p->mask_pitch < 1) return COSA_ERR_INVALID_ARG;
  if (!(p->sm_scale > 0.0) || !std::isfinite(p->sm_scale) || std::isnan(p->skip_delta)) return COSA_ERR_INVALID_ARG;
  if ((p->flags & ~(COSA_FLAG_TEST_STALL | COSA_FLAG_ASCENDING_ORDER | COSA_FLAG_BINARY_MASK | COSA_FLAG_TOP_P |
                    COSA_FLAG_GQA_UNION)) != 0)
    return COSA_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return COSA_ERR_UNSUPPORTED;
  if (p->block_size != 64 && p->block_size != 128) return COSA_ERR_UNSUPPORTED;
  if (p->page_size != 16 && p->page_size != 32 && p->page_size != 64 && p->page_size != 128) return COSA_ERR_UNSUPPORTED;
  if (p->block_size % p->page_size != 0) return COSA_ERR_UNSUPPORTED;
  if (p->max_pages_per_req < ceil_div(p->max_seqlen, p->page_size)) return COSA_ERR_INVALID_ARG;
  return COSA_OK;
}

// Checks of the KAP parameters (stride, budget, mask pitch), shared by the workspace-size query and
// both select calls, so that no size is computed for a problem the calls would refuse.
int check_kap(const cosa_params* p) {
  const int rc = check_common(p);
  if (rc != COSA_OK) return rc;
  if (p->stride < 1 || p->block_size % p->stride != 0) return COSA_ERR_INVALID_ARG;
  const int kb = p->block_size / p->stride;
  if (kb != 4 && kb != 8 && kb != 16) return COSA_ERR_UNSUPPORTED;
  if (p->budget_ppm < 1 || p->budget_ppm > 1000000) return COSA_ERR_INVALID_ARG;
  const int64_t nqb_max = ceil_div(p->max_seqlen, p->block_size);
  if (nqb_max > kMaxQueryBlocksKap) return COSA_ERR_UNSUPPORTED;
  if (p->mask_pitch < ceil_div(static_cast<int64_t>(p->budget_ppm) * nqb_max, 1000000)) return COSA_ERR_INVALID_ARG;
  if ((p->flags & COSA_FLAG_TOP_P) && p->mask_pitch < nqb_max) return COSA_ERR_INVALID_ARG;
  return COSA_OK;
}

}  // namespace

bool cosa::encode_tiled_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                             const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
bool encode_tiled(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                  const cuuint32_t* box) {
  return cosa::encode_tiled_bf16(map, base, rank, dims, strides, box);
}
}  // namespace

extern "C" {

int cosa_version(void) { return (0 << 16) | 1; }

const char* cosa_status_string(int status) {
  switch (status) {
    case COSA_OK: return "ok";
    case COSA_ERR_INVALID_ARG: return "invalid argument";
    case COSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case COSA_ERR_CUDA: return "CUDA launch or driver error";
    case COSA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case COSA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case COSA_ERR_BAD_INPUT: return "cu_seqlens inconsistent with the parameters";
    default: return "unknown status";
  }
}

size_t cosa_proxy_workspace_size(const cosa_params* p) {
  if (check_kap(p) != COSA_OK) return 0;
  return cosa::kap_workspace_bytes(p->num_reqs, p->num_q_heads, p->num_kv_heads, p->block_size, p->stride,
                                   p->total_tokens, p->max_seqlen);
}

int cosa_proxy_select(const cosa_params* p, const void* q, const int32_t* cu_seqlens, const void* k_cache,
                      const int32_t* page_table, int32_t* mask, int32_t* mask_len, void* workspace,
                      size_t workspace_bytes, int32_t* device_status, void* stream) {
  const int rc = check_kap(p);
  if (rc != COSA_OK) return rc;
  if (!q || !cu_seqlens || !k_cache || !page_table || !mask || !mask_len || !workspace) return COSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(cu_seqlens, 4) || !aligned(page_table, 4) ||
      !aligned(mask, 4) || !aligned(mask_len, 4))
    return COSA_ERR_INVALID_ARG;
  const size_t need = cosa_proxy_workspace_size(p);
  if (workspace_bytes < need || !aligned(workspace, 256)) return COSA_ERR_WORKSPACE;
  KapLaunch L{};
  L.q = static_cast<const uint16_t*>(q);
  L.cu_seqlens = cu_seqlens;
  L.k_cache = static_cast<const uint16_t*>(k_cache);
  L.page_table = page_table;
  L.mask = mask;
  L.mask_len = mask_len;
  L.status = device_status;
  L.workspace = workspace;
  L.workspace_bytes = workspace_bytes;
  L.num_reqs = p->num_reqs;
  L.num_q_heads = p->num_q_heads;
  L.num_kv_heads = p->num_kv_heads;
  L.head_dim = p->head_dim;
  L.block_size = p->block_size;
  L.page_size = p->page_size;
  L.stride = p->stride;
  L.total_tokens = p->total_tokens;
  L.max_seqlen = p->max_seqlen;
  L.num_pages = p->num_pages;
  L.max_pages_per_req = p->max_pages_per_req;
  L.mask_pitch = p->mask_pitch;
  L.budget_ppm = p->budget_ppm;
  L.sm_scale = p->sm_scale;
  L.flags = p->flags;
  const cudaError_t e = cosa::launch_kap(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? COSA_OK : COSA_ERR_CUDA;
}

int cosa_proxy_select_static(const cosa_params* p, const void* q, const int32_t* cu_seqlens, const void* k_cache,
                             const int32_t* page_table, int32_t* mask, int32_t* mask_len, int32_t* device_status,
                             void* stream) {
  const int rc = check_kap(p);
  if (rc != COSA_OK) return rc;
  const size_t need = cosa_proxy_workspace_size(p);
  if (need == 0 || need > cosa::kStaticScratchBytes) return COSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (cosa::kap_static_scratch(&scratch) != cudaSuccess) return COSA_ERR_CUDA;
  return cosa_proxy_select(p, q, cu_seqlens, k_cache, page_table, mask, mask_len, scratch, cosa::kStaticScratchBytes,
                           device_status, stream);
}

size_t cosa_prefill_workspace_size(const cosa_params* p) {
  (void)p;
  return 0;
}

int cosa_sparse_prefill(const cosa_params* p, const void* q, const int32_t* cu_seqlens, const void* k_cache,
                        const void* v_cache, const int32_t* page_table, const int32_t* mask,
                        const int32_t* mask_len, void* out, uint8_t* visit_flags, void* workspace,
                        size_t workspace_bytes, int32_t* device_status, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  int rc = check_common(p);
  if (rc != COSA_OK) return rc;
  const int64_t nqb_max = ceil_div(p->max_seqlen, p->block_size);
  if (nqb_max > kMaxQueryBlocksOsk) return COSA_ERR_UNSUPPORTED;
  if ((p->flags & COSA_FLAG_GQA_UNION) && (p->block_size != 128 || (p->flags & COSA_FLAG_BINARY_MASK)))
    return COSA_ERR_UNSUPPORTED;
  if (!q || !cu_seqlens || !k_cache || !v_cache || !page_table || !mask || !mask_len || !out) return COSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens, 4) || !aligned(page_table, 4) || !aligned(mask, 4) || !aligned(mask_len, 4))
    return COSA_ERR_INVALID_ARG;
  if (p->total_tokens == 0) return COSA_OK;
  OskLaunch L{};
  const cuuint64_t d = static_cast<cuuint64_t>(p->head_dim);
  // {d mod 64, row, d / 64, head} views: see OskLaunch
  const cuuint64_t dh = d / 64;
  {
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(p->total_tokens), dh, static_cast<cuuint64_t>(p->num_q_heads)};
    const cuuint64_t strides[3] = {d * 2 * p->num_q_heads, 128, d * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(p->block_size), 1, 1};
    if (!encode_tiled(&L.qmap, q, 4, dims, strides, box)) return COSA_ERR_CUDA;
  }
  {
    const int64_t rows = static_cast<int64_t>(p->num_pages) * p->page_size;
    if (rows > INT32_MAX) return COSA_ERR_UNSUPPORTED;   // TMA coordinates are 32-bit
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), dh, static_cast<cuuint64_t>(p->num_kv_heads)};
    const cuuint64_t strides[3] = {d * 2 * p->num_kv_heads, 128, d * 2};
    const cuuint32_t box_blk[4] = {64, static_cast<cuuint32_t>(p->block_size), static_cast<cuuint32_t>(dh), 1};
    const cuuint32_t box_pg[4] = {64, static_cast<cuuint32_t>(p->page_size), 1, 1};
    if (!encode_tiled(&L.kmap_blk, k_cache, 4, dims, strides, box_blk)) return COSA_ERR_CUDA;
    if (!encode_tiled(&L.kmap_pg, k_cache, 4, dims, strides, box_pg)) return COSA_ERR_CUDA;
    if (!encode_tiled(&L.vmap_blk, v_cache, 4, dims, strides, box_blk)) return COSA_ERR_CUDA;
    if (!encode_tiled(&L.vmap_pg, v_cache, 4, dims, strides, box_pg)) return COSA_ERR_CUDA;
  }
  L.cu_seqlens = cu_seqlens;
  L.page_table = page_table;
  L.mask = mask;
  L.mask_len = mask_len;
  L.out = out;
  L.visit_flags = visit_flags;
  L.status = device_status;
  L.num_reqs = p->num_reqs;
  L.num_q_heads = p->num_q_heads;
  L.num_kv_heads = p->num_kv_heads;
  L.head_dim = p->head_dim;
  L.block_size = p->block_size;
  L.page_size = p->page_size;
  L.total_tokens = p->total_tokens;
  L.max_seqlen = p->max_seqlen;
  L.num_pages = p->num_pages;
  L.max_pages_per_req = p->max_pages_per_req;
  L.mask_pitch = p->mask_pitch;
  L.sm_scale = p->sm_scale;
  L.skip_delta = p->skip_delta;
  L.flags = p->flags;
  const cudaError_t e = cosa::launch_osk(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? COSA_OK : COSA_ERR_CUDA;
}

}  // extern "C"
