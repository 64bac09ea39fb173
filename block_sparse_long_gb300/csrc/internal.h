// Host-side declarations shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace cosa {

constexpr uint8_t kVisitComputed = 0;
constexpr uint8_t kVisitSkipped = 1;
constexpr uint8_t kVisitIgnored = 2;

// bf16 tiled TMA descriptor with 128-byte swizzle (dims/strides innermost first, strides in bytes
// for dims 1..rank-1).  Returns false if the driver entry point is missing or rejects the map.
bool encode_tiled_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box);

// ---------------------------------------------------------------------------
// OSK
// ---------------------------------------------------------------------------
// The TMA maps view a [rows, heads, d] bf16 tensor as {d mod 64, row, d / 64, head} (row stride
// heads * d * 2 bytes, then 128 bytes, then d * 2 bytes), so that one box lands in shared memory as
// [d / 64][rows][128 B], the 128-byte-swizzled K-major layout the tensor cores read.
struct OskLaunch {
  CUtensorMap qmap;      // q [T, Hq, d]: box {64, block_size, 1, 1} (one 64-wide d chunk of a query block)
  CUtensorMap kmap_blk;  // K [pages * P, Hkv, d]: box {64, block_size, d / 64, 1} (a block on consecutive pages)
  CUtensorMap kmap_pg;   // K: box {64, P, 1, 1} (one d chunk of one page)
  CUtensorMap vmap_blk;  // V, as kmap_blk
  CUtensorMap vmap_pg;   // V, as kmap_pg
  const int32_t* cu_seqlens;
  const int32_t* page_table;
  const int32_t* mask;
  const int32_t* mask_len;
  void* out;
  uint8_t* visit_flags;
  int32_t* status;
  int num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, page_size;
  int total_tokens, max_seqlen, num_pages, max_pages_per_req, mask_pitch;
  double sm_scale, skip_delta;
  int flags;             // COSA_FLAG_*
};

size_t osk_smem_bytes(int block_size, int head_dim);
cudaError_t launch_osk(const OskLaunch& L, cudaStream_t stream);

// ---------------------------------------------------------------------------
// KAP
// ---------------------------------------------------------------------------
struct KapLaunch {
  const uint16_t* q;
  const int32_t* cu_seqlens;
  const uint16_t* k_cache;
  const int32_t* page_table;
  int32_t* mask;
  int32_t* mask_len;
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
  int num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, page_size, stride;
  int total_tokens, max_seqlen, num_pages, max_pages_per_req, mask_pitch, budget_ppm;
  double sm_scale;
  int flags;             // COSA_FLAG_*
};

size_t kap_workspace_bytes(int num_reqs, int num_q_heads, int num_kv_heads, int block_size, int stride,
                           int total_tokens, int max_seqlen);

// Fixed device scratch of cosa_proxy_select_static (defined in kap.cu).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxStaticContexts = 64;
// Device address of that scratch in the current context (looked up on the first call per context).
cudaError_t kap_static_scratch(void** ptr);
cudaError_t launch_kap(const KapLaunch& L, cudaStream_t stream);

}  // namespace cosa
