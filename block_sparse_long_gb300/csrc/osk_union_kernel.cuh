// OSK with a GQA page union: one K stream serving two query heads of a kv group.
//
// PageWeaver notes, Sec. 2.2 (the union U_G of a group's selections, the membership mask M_{i,p} and
// the reuse rate rho_Q) applied to the ordered visits of CoSA Sec. 4.3 / Algorithm A
// (ordered-skipping stage).  A work item is a (request, kv head, pair of query heads, query block).
// Its two heads keep their own computation-order masks, visiting orders, running maxima and skip
// votes; what they share is the K traffic.  The K producer merges the two ordered, de-duplicated
// block lists into one stream: at every step it loads the block that is next for both heads if
// they agree, otherwise the lower of the two next blocks, which serves only the head it is next
// for.  Each head therefore sees exactly its own sequence, in its own order, and every block that
// both heads want at the same point of their walks is gathered once.
//
// Warp roles (352 threads):
//   warps 0-3    head 0 of the pair; warps 4-7 head 1.  Thread t of a group owns row t (TMEM lane
//                t), all b columns: per visit it reads S in two 64-column loads, applies the masks,
//                votes on the skip (Eq. (5)) within its group, and for computed blocks writes
//                P = exp(S - m_ref) as bf16 over the first b/2 columns of its own S buffer.  The
//                group's first thread also gathers V of the computed block (requested right after
//                the vote) and issues O_h += P_h V once every P is written.
//   warp 8       K producer: both mask rows (invalid and repeated IDs dropped, first occurrence
//                kept), the merge, the page table, the TMA gathers of the stream's K tiles.
//   warps 9/10   S issuers of head 0 / head 1 (warp 9 owns TMEM): S_h = Q_h K^T for every stream
//                block the head is a member of.
//
// Tensor memory (512 columns): S of head 0 and 1 (b columns each), O of head 0 and 1 (d columns
// each).  With one S buffer per head, a head's next product waits for the vote on its previous
// block (skipped) or for its P.V (computed), so the head's V slot and O are never busy when its
// softmax reaches a computed block; the two heads' chains run side by side.
//
// Per head, the arithmetic is that of osk_kernel: the same products, the same order of visits,
// the same fp32 operations in the same order (row maxima, the skip test, exponentials, the row
// sums of the two column halves, the lazy rescale), so outputs and visit flags equal that
// kernel's bit for bit.
#pragma once
#include "osk_kernel.cuh"

namespace cosa {
namespace {

constexpr int kUThreads = 352;
constexpr int kUWarpK = 8, kUWarpS0 = 9, kUWarpS1 = 10;
constexpr uint32_t kUSharedBit = 1u << 16;  // in KInfo::pages of a head's visit record: K loaded for both heads

// one entry of the merged K stream
struct alignas(16) UInfo {
  int32_t blk;       // block id, -1 = end of the item
  uint32_t pages;    // bit u set: page u of the block exists
  int32_t kk[2];     // index of the entry in each member head's mask row
  int32_t kvh;
  int32_t members;   // bit x: head x of the pair visits this block now
  int32_t pad[2];
  int32_t phys[kMaxPagesPerBlock];
};

template <int HD>
struct alignas(1024) UnionSmem {
  static constexpr int BLK = 128;
  static constexpr int NK = (HD == 64) ? 4 : 2;
  static constexpr int TILE = BLK * HD * 2;
  static constexpr int HALF = BLK * 128;
  uint8_t q[2][128 * HD * 2];   // Q of each head, [HD/64][128 rows][128 B], SW128
  uint8_t k[NK][TILE];
  uint8_t v[2][TILE];           // V of each head's current computed block; its output staging tile
  uint64_t q_full, q_free;
  uint64_t k_full[NK], k_free[NK];
  uint64_t s_full[2], s_free[2];
  uint64_t v_full[2];
  uint64_t o_done[2][2];
  uint64_t cleanup;
  UInfo info[8];                // stream entry e in slot e & 7
  KInfo hrec[2][8];             // head x's visit vx in slot vx & 7 (written by its S issuer)
  KInfo stage[2][32];           // the producer's kept entries of each head, in mask order
  uint32_t tmem_base;
  int32_t abort_flag;
  alignas(4) uint8_t stopf[2][2][4];   // [head][visit & 1][softmax warp]: 0 go on, 1 stop, 2 a wait ran out
  uint32_t seen[2][kMaxBlocksPerReq / 32];
};

// Work item `idx`: kv-head major, heaviest query blocks first, then requests, then head pairs.
struct PairItem {
  int b, h[2], kvh, i, tok0, L, nblk;
  int state;  // 0 run, 1 absent query block, 2 bad cu_seqlens
};

__device__ __forceinline__ PairItem decode_pair(const OskArgs& a, int idx) {
  PairItem it;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int G2 = (G + 1) / 2;
  const int pr = idx % G2;
  idx /= G2;
  it.b = idx % a.num_reqs;
  idx /= a.num_reqs;
  it.i = a.nqb_max - 1 - (idx % a.nqb_max);
  it.kvh = idx / a.nqb_max;
  it.h[0] = it.kvh * G + 2 * pr;
  it.h[1] = (2 * pr + 1 < G) ? it.h[0] + 1 : -1;
  it.tok0 = a.cu_seqlens[it.b];
  it.L = a.cu_seqlens[it.b + 1] - it.tok0;
  it.nblk = (it.L + 127) / 128;
  if (it.L < 0 || it.L > a.max_seqlen || it.tok0 < 0 || it.tok0 + it.L > a.total_tokens) it.state = 2;
  else it.state = (it.i >= it.nblk) ? 1 : 0;
  return it;
}

template <int HD, int PSZ, bool SKIP, bool FLAGS>
__global__ void __launch_bounds__(kUThreads, 1)
    osk_union_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap_blk,
                     const __grid_constant__ CUtensorMap kmap_pg, const __grid_constant__ CUtensorMap vmap_blk,
                     const __grid_constant__ CUtensorMap vmap_pg, const OskArgs a) {
  using S = UnionSmem<HD>;
  constexpr int BLK = 128;
  constexpr int NK = S::NK;
  constexpr int DH = HD / 64;
  constexpr int P = PSZ;
  constexpr int pages_per_blk = BLK / P;
  constexpr uint32_t all_pages = (1u << pages_per_blk) - 1u;
  static_assert(BLK % P == 0 && pages_per_blk <= kMaxPagesPerBlock, "a block is whole pages");
  static_assert(S::TILE >= 128 * HD * 2, "a V slot stages one output tile");
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  volatile int* abort_flag = &sm.abort_flag;

  // ---------------- set-up (once per CTA) ----------------
  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, 2);          // one commit from each S issuer
    for (int s = 0; s < NK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_free[s], 2);     // each S issuer: its product's commit, or a plain arrive
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.s_full[x], 2);     // plain arrive (visit record) + product commit
      mbar_init(&sm.s_free[x], 1);     // the vote (skipped, end) or the P.V commit (computed)
      mbar_init(&sm.v_full[x], 1);
      mbar_init(&sm.o_done[x][0], 1);
      mbar_init(&sm.o_done[x][1], 1);
    }
    mbar_init(&sm.cleanup, 4);         // both S issuers and both heads' P.V issuers
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kUWarpS0) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kUWarpK) {
    // =========================== K producer ===========================
    const uint32_t lane = lane_id();
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap_blk);
      tma_prefetch_desc(&kmap_pg);
      tma_prefetch_desc(&vmap_blk);
      tma_prefetch_desc(&vmap_pg);
    }
    int e = 0, n = 0;   // stream entries (all items), items
    bool ok = !a.stall;
    for (int idx = blockIdx.x; idx < a.num_items && ok; idx += gridDim.x) {
      const PairItem it = decode_pair(a, idx);
      if (it.state == 2 && lane == 0) report_status(a.status, kStatusBadInput);
      if (it.state != 0) continue;
      const int i = it.i, nblk = it.nblk, kvh = it.kvh;
      const int nh = (it.h[1] >= 0) ? 2 : 1;
      const int req_pages = (it.L + P - 1) / P;
      const int32_t* pt_row = a.page_table + static_cast<size_t>(it.b) * a.max_pages_per_req;
      const int32_t* mask_row[2] = {nullptr, nullptr};
      uint8_t* flags_row[2] = {nullptr, nullptr};
      int n_entries[2] = {0, 0};
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (x >= nh) break;
        const size_t row_base = (static_cast<size_t>(it.b) * a.num_q_heads + it.h[x]) * a.nqb_max + i;
        mask_row[x] = a.mask + row_base * a.mask_pitch;
        if (FLAGS) flags_row[x] = a.visit_flags + row_base * a.mask_pitch;
        const int ne = a.mask_len[row_base];
        n_entries[x] = ne < 0 ? 0 : (ne > a.mask_pitch ? a.mask_pitch : ne);
        for (int w = lane; w < (nblk + 31) / 32; w += 32) sm.seen[x][w] = 0u;
        if (FLAGS)
          for (int k = n_entries[x] + lane; k < a.mask_pitch; k += 32) flags_row[x][k] = kVisitIgnored;
      }
      __syncwarp();
      // Q of both heads, once every product of the previous item has completed
      if (n > 0) ok = warp_wait(&sm.q_free, (n - 1) & 1, abort_flag, a.status);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full, static_cast<uint32_t>(nh) * BLK * HD * 2);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (x >= nh) break;
          for (int dh = 0; dh < DH; ++dh)
            tma_load_4d(&sm.q[x][dh * 128 * 128], &qmap, &sm.q_full, 0, it.tok0 + i * BLK, dh, it.h[x]);
        }
      }
      ++n;
      // staged kept entries of each head: cnt staged, cur consumed, scan = next mask entry to read
      int cnt[2] = {0, 0}, cur[2] = {0, 0}, scan[2] = {0, 0};
      while (ok) {
        // refill the stage of a head whose staged entries are all consumed
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (x >= nh) break;
          while (cur[x] == cnt[x] && scan[x] < n_entries[x]) {
            const int k = scan[x] + static_cast<int>(lane);
            const int j = (k < n_entries[x]) ? mask_row[x][k] : -1;
            const bool valid = (k < n_entries[x]) && j >= 0 && j <= i && j < nblk;
            const unsigned peers = __match_any_sync(0xffffffffu, valid ? j : -1 - static_cast<int>(lane));
            const bool first = valid && (static_cast<int>(lane) == __ffs(peers) - 1);
            const bool dup = first && ((sm.seen[x][j >> 5] >> (j & 31)) & 1u);
            const bool keep = first && !dup;
            __syncwarp();
            if (keep) atomicOr(&sm.seen[x][j >> 5], 1u << (j & 31));
            if (FLAGS && k < n_entries[x] && !keep) flags_row[x][k] = kVisitIgnored;
            const unsigned kept = __ballot_sync(0xffffffffu, keep);
            if (keep) {
              KInfo& st = sm.stage[x][__popc(kept & ((1u << lane) - 1u))];
              uint32_t pages = 0;
#pragma unroll
              for (int u = 0; u < kMaxPagesPerBlock; ++u) {
                int ph = -1;
                if (u < pages_per_blk) {
                  const int lp = j * pages_per_blk + u;
                  const int pp = (lp < req_pages) ? pt_row[lp] : -1;
                  if (pp >= 0 && pp < a.num_pages) { ph = pp; pages |= 1u << u; }
                }
                st.phys[u] = ph;
              }
              st.blk = j;
              st.pages = pages;
              st.k = k;
              st.kvh = kvh;
            }
            __syncwarp();
            cnt[x] = __popc(kept);
            cur[x] = 0;
            scan[x] += 32;
          }
        }
        const bool has0 = cur[0] < cnt[0];
        const bool has1 = (nh > 1) && cur[1] < cnt[1];
        if (!has0 && !has1) break;
        // the merge: the block both heads want next, else the lower of the two next blocks
        const int j0 = has0 ? sm.stage[0][cur[0]].blk : 0x7fffffff;
        const int j1 = has1 ? sm.stage[1][cur[1]].blk : 0x7fffffff;
        const int members = (j0 <= j1 ? 1 : 0) | (j1 <= j0 ? 2 : 0);
        const int slot = e % NK;
        if (e >= NK) ok = warp_wait(&sm.k_free[slot], ((e / NK) - 1) & 1, abort_flag, a.status);
        if (!ok) break;
        if (lane == 0) {
          const KInfo& st = (members & 1) ? sm.stage[0][cur[0]] : sm.stage[1][cur[1]];
          UInfo& ui = sm.info[e & 7];
          ui.blk = st.blk;
          ui.pages = st.pages;
          ui.kk[0] = (members & 1) ? sm.stage[0][cur[0]].k : -1;
          ui.kk[1] = (members & 2) ? sm.stage[1][cur[1]].k : -1;
          ui.kvh = kvh;
          ui.members = members;
#pragma unroll
          for (int u = 0; u < kMaxPagesPerBlock; ++u) ui.phys[u] = st.phys[u];
          if (pages_consecutive(st.pages, all_pages, st.phys, pages_per_blk)) {
            mbar_arrive_expect_tx(&sm.k_full[slot], BLK * HD * 2);
            tma_load_4d(&sm.k[slot][0], &kmap_blk, &sm.k_full[slot], 0, st.phys[0] * P, 0, kvh);
          } else {
            const uint32_t bytes = static_cast<uint32_t>(__popc(st.pages)) * DH * P * 128u;
            mbar_arrive_expect_tx(&sm.k_full[slot], bytes);
            for (int u = 0; u < pages_per_blk; ++u) {
              if (!((st.pages >> u) & 1u)) continue;
              for (int dh = 0; dh < DH; ++dh)
                tma_load_4d(&sm.k[slot][dh * S::HALF + u * P * 128], &kmap_pg, &sm.k_full[slot], 0, st.phys[u] * P, dh,
                            kvh);
            }
          }
        }
        __syncwarp();
        ++e;
        if (members & 1) ++cur[0];
        if (members & 2) ++cur[1];
      }
      // end of the item, for every head of the pair
      if (ok) {
        const int slot = e % NK;
        if (e >= NK) ok = warp_wait(&sm.k_free[slot], ((e / NK) - 1) & 1, abort_flag, a.status);
        if (ok && lane == 0) {
          sm.info[e & 7].blk = -1;
          sm.info[e & 7].members = (nh > 1) ? 3 : 1;
          mbar_arrive(&sm.k_full[slot]);
        }
        __syncwarp();
        ++e;
      }
    }
    // on abort, let every issued copy land before the CTA exits
    if (*abort_flag && lane == 0) {
      if (n > 0) wait_parity_bounded(&sm.q_full, (n - 1) & 1, nullptr, nullptr);
      for (int s = 0; s < NK; ++s) {
        const int issued = (e > s) ? (e - s + NK - 1) / NK : 0;
        if (issued > 0) wait_parity_bounded(&sm.k_full[s], (issued - 1) & 1, nullptr, nullptr);
      }
    }
  } else if (warp == kUWarpS0 || warp == kUWarpS1) {
    // =========================== S issuers (lane 0 of two warps) ===========================
    // Issuer X walks every stream entry: K(e) has landed, then, if head X is a member, S_X = Q_X K^T
    // once the head's previous visit has released S_X; the K slot is released by the product's
    // commit, or at once if X is not a member (so no issuer falls a phase behind on a slot).
    if (lane_id() == 0) {
      const int X = (warp == kUWarpS0) ? 0 : 1;
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BLK, false, false);
      const uint64_t qdesc = smem_desc_sw128(smem_u32(&sm.q[X][0]), 16, 1024);
      const uint64_t kdesc = smem_desc_sw128(smem_u32(&sm.k[0][0]), 16, 1024);
      int e = 0, vx = 0, n = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < a.num_items && ok; idx += gridDim.x) {
        const PairItem it = decode_pair(a, idx);
        if (it.state != 0) continue;
        ok = wait_parity_bounded(&sm.q_full, n & 1, abort_flag, a.status);
        ++n;
        tc_fence_after();
        while (ok) {
          const int slot = e % NK;
          if (!wait_parity_bounded(&sm.k_full[slot], (e / NK) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          // info[e & 7] is rewritten with entry e + 8, after both issuers have passed e + 8 - NK
          const UInfo& ui = sm.info[e & 7];
          const int blk = ui.blk;
          const bool mine = (ui.members >> X) & 1;
          if (mine) {
            if (vx > 0 && !wait_parity_bounded(&sm.s_free[X], (vx - 1) & 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            KInfo& hr = sm.hrec[X][vx & 7];
            hr.blk = blk;
            hr.pages = ui.pages | ((ui.members == 3) ? kUSharedBit : 0u);
            hr.k = ui.kk[X];
            hr.kvh = ui.kvh;
#pragma unroll
            for (int u = 0; u < kMaxPagesPerBlock; ++u) hr.phys[u] = ui.phys[u];
            mbar_arrive(&sm.s_full[X]);
            ++vx;
          }
          if (blk < 0) {
            // end of the item: no product; S_X (if a member) and the K slot pass on unused
            if (mine) mbar_arrive(&sm.s_full[X]);
            mbar_arrive(&sm.k_free[slot]);
            ++e;
            break;
          }
          if (mine) {
            tc_fence_after();
            const uint64_t kslot = kdesc + static_cast<uint64_t>(slot * (S::TILE >> 4));
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const uint64_t ad = qdesc + static_cast<uint64_t>(((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4);
              const uint64_t bd = kslot + static_cast<uint64_t>(((kk >> 2) * S::HALF + (kk & 3) * 32) >> 4);
              umma_ss(tmem + X * 128u, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(&sm.s_full[X]);
            umma_commit(&sm.k_free[slot]);
          } else {
            mbar_arrive(&sm.k_free[slot]);
          }
          ++e;
        }
        // Q may be replaced once this issuer's products of the item have completed
        if (ok) umma_commit(&sm.q_free);
      }
      umma_commit(&sm.cleanup);
      wait_parity_bounded(&sm.cleanup, 0, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // =========================== softmax of one head (4 warps) ===========================
    const int X = warp >> 2;                // head of the pair
    const int t = (warp & 3) * 32 + static_cast<int>(lane_id());   // tile row == TMEM lane
    const uint32_t lane = lane_id();
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t bar_stop = 1 + 4 * X, bar_vote = 2 + 4 * X, bar_epi = 3 + 4 * X, bar_p = 4 + 4 * X;
    const uint32_t sbase = tmem + lane_addr + X * 128u;             // S_X (P over its first b/2 columns)
    const uint32_t obase = tmem + lane_addr + 256u + X * HD;        // O_X
    constexpr bool use_skip = SKIP;
    const float sl2 = a.scale_log2;
    constexpr int pshift = (P == 16) ? 4 : (P == 32) ? 5 : (P == 64) ? 6 : 7;
    const bool lead_warp = (warp & 3) == 0;
    const bool leader = lead_warp && lane == 0;
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD, false, true);
    const uint64_t vdesc = smem_desc_sw128(smem_u32(&sm.v[X][0]), S::HALF, 1024);
    int vx = 0;                // this head's visits, all items
    int c = 0;                 // this head's computed visits (= V loads), all items
    bool ok = true;
    bool local_fail = false;
    for (int idx = blockIdx.x; idx < a.num_items && ok; idx += gridDim.x) {
      const PairItem it = decode_pair(a, idx);
      const int hX = X ? it.h[1] : it.h[0];
      if (it.state != 0 || hX < 0) continue;
      const int i = it.i, L = it.L;
      const int pos = i * BLK + t;
      const bool row_valid = pos < L;
      const float tau2 = use_skip ? log2f(static_cast<float>(a.skip_delta)) - log2f(static_cast<float>(L)) : 0.0f;
      const size_t row_base = (static_cast<size_t>(it.b) * a.num_q_heads + hX) * a.nqb_max + i;
      uint8_t* flags_row = FLAGS ? a.visit_flags + row_base * a.mask_pitch : nullptr;
      float m_run = -INFINITY, m_ref = -INFINITY;
      float l_half[2] = {0.0f, 0.0f};   // row sums of columns [0, b/2) and [b/2, b), as osk_kernel keeps them
      int c_item = 0;
      for (;; ++vx) {
        int ki_blk = -1, ki_k = 0;
        uint32_t ki_pages = 0;
        bool shared = false;
        float pm[2] = {-INFINITY, -INFINITY};   // row max of each column half
        bool okw = !local_fail && wait_parity_bounded(&sm.s_full[X], vx & 1, abort_flag, a.status);
        okw = __all_sync(0xffffffffu, okw);
        bool need_mask = false;
        int lim = -1;
        if (okw) {
          // hrec[X][vx & 7] is rewritten at visit vx + 8, after this visit has released S_X
          const int4 hd = *reinterpret_cast<const int4*>(&sm.hrec[X][vx & 7]);
          ki_blk = hd.x;
          ki_pages = static_cast<uint32_t>(hd.y) & 0xffffu;
          shared = (static_cast<uint32_t>(hd.y) & kUSharedBit) != 0;
          ki_k = hd.z;
          if (ki_blk >= 0) {
            const int key0 = ki_blk * BLK;
            need_mask = (ki_blk == i) || (key0 + BLK > L) || (ki_pages != all_pages) || !row_valid;
            lim = row_valid ? min(pos, L - 1) - key0 : -1;  // last visible column
            tc_fence_after();
            // each column half's maximum, from the load itself unless masked columns must leave it
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t r[64];
              float mx;
              tmem_ld64_max(sbase + hh * 64, r, mx);
              tmem_wait_ld();
              reg_after_wait(mx);
              if (need_mask) {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int q = 0; q < 64; ++q) {
                  const int col = hh * 64 + q;
                  const bool vis = col <= lim && ((ki_pages >> (col >> pshift)) & 1u);
                  if (vis) m4[q & 3] = fmaxf(m4[q & 3], __uint_as_float(r[q]));
                }
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
              }
              pm[hh] = mx;
            }
            tc_fence_before();
          }
        }
        // skip vote (Eq. (5)): a row wants the block iff m_loc - max(m_run, m_loc) >= tau2, which is
        // monotone in m_loc, so testing each half's maximum decides as the row maximum does
        const float p0 = (pm[0] == -INFINITY) ? -INFINITY : pm[0] * sl2;
        const float p1 = (pm[1] == -INFINITY) ? -INFINITY : pm[1] * sl2;
        bool want = true;
        if (use_skip) {
          const bool w0 = (p0 != -INFINITY) && (p0 - fmaxf(m_run, p0) >= tau2);
          const bool w1 = (p1 != -INFINITY) && (p1 - fmaxf(m_run, p1) >= tau2);
          want = row_valid && (w0 || w1);
        }
        // each warp's stop code goes to shared memory before the vote and is read after it: one
        // barrier decides the visit (compute, skip, end of the item, or a wait ran out)
        const bool stop = !okw || (ki_blk < 0);
        if (lane == 0) sm.stopf[X][vx & 1][warp & 3] = stop ? (okw ? 1 : 2) : 0;
        const bool compute = named_bar_red_or(bar_vote, 128, want || stop);
        const uint32_t stops = compute ? *reinterpret_cast<const volatile uint32_t*>(&sm.stopf[X][vx & 1][0]) : 0u;
        if (stops != 0) {
          if (stops & 0x02020202u) ok = false;
          // the end of the item releases S_X for the next item's first product
          if (ok && leader) mbar_arrive(&sm.s_free[X]);
          ++vx;
          break;
        }
        if (!compute) {
          // every warp of the head has read S_X (the vote barrier orders the loads before this)
          if (leader) {
            mbar_arrive(&sm.s_free[X]);
            if (flags_row) flags_row[ki_k] = kVisitSkipped | (shared ? 4 : 0);
          }
          continue;
        }
        const float mx = fmaxf(pm[0], pm[1]);
        const float m_loc = (mx == -INFINITY) ? -INFINITY : mx * sl2;
        const float m_new = fmaxf(m_run, m_loc);
        m_run = m_new;
        if (lead_warp) {
          // V of this block into the head's V slot (idle: the previous P.V completed before S_X was
          // refilled); rows of pages that do not exist are zero, since 0 * V must stay 0
          const KInfo& r = sm.hrec[X][vx & 7];
          if (ki_pages != all_pages) {
            for (int u = 0; u < pages_per_blk; ++u) {
              if ((ki_pages >> u) & 1u) continue;
              for (int dh = 0; dh < DH; ++dh) {
                uint4* z = reinterpret_cast<uint4*>(&sm.v[X][dh * S::HALF + u * P * 128]);
                for (int q = lane; q < P * 8; q += 32) z[q] = make_uint4(0, 0, 0, 0);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            if (flags_row) flags_row[ki_k] = kVisitComputed | (shared ? 4 : 0);
            if (pages_consecutive(ki_pages, all_pages, r.phys, pages_per_blk)) {
              mbar_arrive_expect_tx(&sm.v_full[X], BLK * HD * 2);
              tma_load_4d(&sm.v[X][0], &vmap_blk, &sm.v_full[X], 0, r.phys[0] * P, 0, r.kvh);
            } else {
              const uint32_t bytes = static_cast<uint32_t>(__popc(ki_pages)) * DH * P * 128u;
              mbar_arrive_expect_tx(&sm.v_full[X], bytes);
              for (int u = 0; u < pages_per_blk; ++u) {
                if (!((ki_pages >> u) & 1u)) continue;
                for (int dh = 0; dh < DH; ++dh)
                  tma_load_4d(&sm.v[X][dh * S::HALF + u * P * 128], &vmap_pg, &sm.v_full[X], 0, r.phys[u] * P, dh,
                              r.kvh);
              }
            }
          }
          __syncwarp();
        }
        const bool first_mass = (m_ref == -INFINITY) && (m_new != -INFINITY);
        const bool rescale = (m_ref != -INFINITY) && (m_new > m_ref + kRescaleLog2);
        float alpha = 1.0f;
        if (first_mass) m_ref = m_new;
        if (rescale) {
          alpha = ex2_approx(m_ref - m_new);
          m_ref = m_new;
          l_half[0] *= alpha;
          l_half[1] *= alpha;
        }
        // P = exp2(S * scale * log2(e) - m_ref) as bf16 pairs over the first b/2 columns of S_X, 32 S
        // columns at a time: the P of columns [32 c, 32 c + 32) goes to [16 c, 16 c + 16), which only
        // holds S columns already read.  Masked entries are -inf -> 0.  Each half's row sum keeps the
        // pairing and order of osk_kernel's column halves.
        const float base = (m_ref == -INFINITY) ? 0.0f : m_ref;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            const int col0 = hh * 64 + hc * 32;
            uint32_t r[32];
            tmem_ld32(sbase + col0, r);
            tmem_wait_ld();
            float sv[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              sv[q] = __uint_as_float(r[q]);
              if (need_mask) {
                const int col = col0 + q;
                if (col > lim || !((ki_pages >> (col >> pshift)) & 1u)) sv[q] = -INFINITY;
              }
            }
            uint32_t pk[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              float x0, x1;
              fma2_bc(x0, x1, sv[2 * q], sv[2 * q + 1], sl2, -base);
              const float e0 = ex2_approx(x0);
              const float e1 = ex2_approx(x1);
              add2_acc(rs4[(q & 1) * 2], rs4[(q & 1) * 2 + 1], e0, e1);
              pk[q] = pack_bf16x2(e0, e1);
            }
            tmem_st16(sbase + col0 / 2, pk);
          }
          l_half[hh] += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        }
        tmem_wait_st();
        // O is scaled once the head's previous P.V has landed; this visit's P.V is issued after the
        // group's barrier below, so it accumulates onto the scaled O
        if (__any_sync(0xffffffffu, rescale) && c_item > 0) {
          bool okr = wait_parity_bounded(&sm.o_done[X][(c - 1) & 1], ((c - 1) >> 1) & 1, abort_flag, a.status);
          if (!__all_sync(0xffffffffu, okr)) { local_fail = true; }
          if (!local_fail) {
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < HD / 16; ++cc) {
              uint32_t r[16];
              tmem_ld16(obase + cc * 16, r);
              tmem_wait_ld();
#pragma unroll
              for (int q = 0; q < 16; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * alpha);
              tmem_st16(obase + cc * 16, r);
              tmem_wait_st();
            }
          }
        }
        // every P (and scaled O) of the group is in TMEM: the first thread issues O += P V once V landed
        tc_fence_before();
        const bool pv_fail = named_bar_red_or(bar_p, 128, local_fail);
        if (leader && !pv_fail) {
          if (wait_parity_bounded(&sm.v_full[X], c & 1, abort_flag, a.status)) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BLK / 16; ++kk) {
              const uint64_t bd = vdesc + static_cast<uint64_t>((kk * 16 * 128) >> 4);
              umma_ts(tmem + 256u + X * HD, tmem + X * 128u + kk * 8, bd, idesc_pv, (c_item > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&sm.s_free[X]);
            umma_commit(&sm.o_done[X][c & 1]);
          }
        }
        if (pv_fail) local_fail = true;
        ++c;
        ++c_item;
      }
      if (!ok) break;
      // ---------------- epilogue: O / l -> bf16 -> global ----------------
      if (c_item > 0) ok = wait_parity_bounded(&sm.o_done[X][(c - 1) & 1], ((c - 1) >> 1) & 1, abort_flag, a.status);
      ok = named_bar_red_or(bar_stop, 128, !ok) ? false : ok;
      if (!ok) break;
      tc_fence_after();
      const float l_sum = l_half[0] + l_half[1];
      const float inv_l = (l_sum > 0.0f) ? 1.0f / l_sum : 0.0f;
      // head X's V slot is idle here: its P.V products are done, the next V load follows the next
      // item's first vote of this head
      uint8_t* stage = &sm.v[X][0];
      constexpr int CH = HD / 8;  // 16-byte chunks per output row
      {
        const uint32_t ob = obase;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          uint32_t r[32];
          if (c_item > 0) {
            tmem_ld32(ob + cc * 32, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) r[q] = 0u;
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * inv_l, __uint_as_float(r[q4 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * inv_l, __uint_as_float(r[q4 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * inv_l, __uint_as_float(r[q4 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * inv_l, __uint_as_float(r[q4 * 8 + 7]) * inv_l);
            const int chunk = cc * 4 + q4;
            const int phys_chunk = chunk ^ (t & (CH - 1));
            *reinterpret_cast<uint4*>(stage + t * (HD * 2) + phys_chunk * 16) = w;
          }
        }
      }
      tc_fence_before();
      named_bar_sync(bar_epi, 128);
      {
        const int rows = min(BLK, L - i * BLK);
        uint8_t* out = reinterpret_cast<uint8_t*>(a.out);
        for (int q = t; q < rows * CH; q += 128) {
          const int r = q / CH, chunk = q % CH;
          const uint4 w = *reinterpret_cast<const uint4*>(stage + r * (HD * 2) + ((chunk ^ (r & (CH - 1))) * 16));
          const size_t tok = static_cast<size_t>(it.tok0) + static_cast<size_t>(i) * BLK + r;
          *reinterpret_cast<uint4*>(out + ((tok * a.num_q_heads + hX) * HD) * 2 + chunk * 16) = w;
        }
      }
      // the staging reads finish before a later TMA load may refill the V slot
      fence_proxy_async_smem();
      named_bar_sync(bar_epi, 128);
    }
    // every P.V issued by this thread completes before TMEM is released; on abort, the last V
    // copy (if any) lands before the CTA exits
    if (leader) {
      umma_commit(&sm.cleanup);
      wait_parity_bounded(&sm.cleanup, 0, nullptr, nullptr);
      if (*abort_flag && c > 0) wait_parity_bounded(&sm.v_full[X], (c - 1) & 1, nullptr, nullptr);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kUWarpS0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int HD, int PSZ, bool SKIP, bool FLAGS>
cudaError_t launch_osk_union_b(const OskLaunch& L, cudaStream_t stream) {
  OskArgs a;
  a.cu_seqlens = L.cu_seqlens;
  a.page_table = L.page_table;
  a.mask = L.mask;
  a.mask_len = L.mask_len;
  a.out = reinterpret_cast<uint16_t*>(L.out);
  a.visit_flags = L.visit_flags;
  a.status = L.status;
  a.num_reqs = L.num_reqs;
  a.num_q_heads = L.num_q_heads;
  a.num_kv_heads = L.num_kv_heads;
  a.total_tokens = L.total_tokens;
  a.max_seqlen = L.max_seqlen;
  a.nqb_max = (L.max_seqlen + 127) / 128;
  a.page_size = L.page_size;
  a.num_pages = L.num_pages;
  a.max_pages_per_req = L.max_pages_per_req;
  a.mask_pitch = L.mask_pitch;
  a.scale_log2 = static_cast<float>(L.sm_scale * 1.4426950408889634);
  a.skip_delta = L.skip_delta;
  a.stall = (L.flags & COSA_FLAG_TEST_STALL) ? 1 : 0;
  const size_t smem = sizeof(UnionSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(osk_union_kernel<HD, PSZ, SKIP, FLAGS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int G = L.num_q_heads / L.num_kv_heads;
  const long long items = static_cast<long long>(L.num_kv_heads) * a.nqb_max * L.num_reqs * ((G + 1) / 2);
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.num_items = static_cast<int>(items);
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  osk_union_kernel<HD, PSZ, SKIP, FLAGS>
      <<<grid, kUThreads, smem, stream>>>(L.qmap, L.kmap_blk, L.kmap_pg, L.vmap_blk, L.vmap_pg, a);
  return cudaGetLastError();
}

template <int HD, int PSZ>
cudaError_t launch_osk_union_s(const OskLaunch& L, cudaStream_t stream) {
  const bool skip = L.skip_delta > 0.0, flags = L.visit_flags != nullptr;
  if (skip)
    return flags ? launch_osk_union_b<HD, PSZ, true, true>(L, stream) : launch_osk_union_b<HD, PSZ, true, false>(L, stream);
  return flags ? launch_osk_union_b<HD, PSZ, false, true>(L, stream) : launch_osk_union_b<HD, PSZ, false, false>(L, stream);
}

template <int HD>
cudaError_t launch_osk_union_hd(const OskLaunch& L, cudaStream_t stream) {
  switch (L.page_size) {
    case 16: return launch_osk_union_s<HD, 16>(L, stream);
    case 32: return launch_osk_union_s<HD, 32>(L, stream);
    case 64: return launch_osk_union_s<HD, 64>(L, stream);
    case 128: return launch_osk_union_s<HD, 128>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_osk_union_d64(const OskLaunch& L, cudaStream_t stream);
cudaError_t launch_osk_union_d128(const OskLaunch& L, cudaStream_t stream);

}  // namespace cosa
