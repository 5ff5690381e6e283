// launch.h -- host-side launchers shared between the translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace psf {

struct FwdParams;
struct BwdParams;

// Forward preparation in one launch: the heaviest-first list of (segment, query
// tile) items (validating the segment arrays; n_items[1] is zeroed as the
// counter of kernels that take items dynamically), and out = 0 / lse = -inf for
// query rows at or past cu_q[nseg].
cudaError_t launch_fwd_prep(const SegInfo& g, int2* items, int* n_items, int* seg_prefix, int item_cap, int* status,
                            void* out, int64_t o_sb, int64_t o_ss, int64_t o_sh, float* lse, int64_t l_sb,
                            int64_t l_sh, int Hq, int Dv, cudaStream_t st);
// Backward work list in the workspace: items (segment, key tile, first step,
// end step), heaviest first, with item_slot[i] the dK/dV partial-sum slot of
// item i (-1: its key tile is whole); splits lists the cut key tiles as
// (first key row, key rows, first slot, slot count). n_items[0] = items, n_items[1]
// the work counter of kernels that take items dynamically, n_items[2] = cut
// tiles.
struct BwdSchedule {
  int4* items;
  int* item_slot;
  int4* splits;
  int* n_items;
  int* seg_prefix;
  int item_cap;
  int slot_cap;
  int nctas;  // CTAs of the attention kernel the list is for
};
// Backward preparation in one launch: the work list (key tiles cut into
// sub-ranges when split_target > 0; n_items[1] zeroed); Delta = rowsum(dO * O)
// (fp32, [Hq][rows]; dO and O each with their own element strides); the zeroed
// dQ accumulator; zeroed dK / dV rows at or past cu_k[nseg].
cudaError_t launch_bwd_prep(const SegInfo& g, int G, int Hkv, int split_target, const BwdSchedule& sc, int* status,
                            const void* dout, int64_t d_sb, int64_t d_ss, int64_t d_sh, const void* out, int64_t o_sb,
                            int64_t o_ss, int64_t o_sh, float* delta, float* dq_acc, int Hq, int Dqk, int Dv, void* dk,
                            void* dv, int64_t k_sb, int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss,
                            int64_t v_sh, int f16, cudaStream_t st);
// Grid: one CTA per SM (two for head dims 64 and 128), at most max_work.
// f16 selects fp16 inputs and outputs (else bf16).
cudaError_t launch_fwd(const FwdParams& p, int dqk, int dvc, int sms, int64_t max_work, int f16, cudaStream_t st);
// The softcapped kernels (fwd_cap.cu); launch_fwd calls it when p.softcap > 0.
cudaError_t launch_fwd_capped(const FwdParams& p, int dqk, int dvc, int grid, int f16, cudaStream_t st);
cudaError_t launch_bwd(const BwdParams& p, int dqk, int dv, int sms, int item_cap, int f16, cudaStream_t st);
// The softcapped kernels (bwd_cap.cu); launch_bwd calls it when p.softcap > 0.
cudaError_t launch_bwd_capped(const BwdParams& p, int dqk, int dv, int grid, int f16, cudaStream_t st);
// Packed query heads (bwd_pack.cu); launch_bwd calls it when p.pack > 1.
cudaError_t launch_bwd_packed(const BwdParams& p, int dqk, int dv, int grid, int f16, cudaStream_t st);
int fwd_smem_bytes(int dqk, int dvc);
int bwd_smem_bytes(int dqk, int dv);

cudaError_t launch_chunk_dense_flags(const int32_t* ids, int B, int S, int q0, int Lq, int k0, int Lk, int32_t* flags,
                                     cudaStream_t st);
cudaError_t launch_build_segments(const int32_t* ids, int B, int Sk, int Lq, int q0, int32_t* cu_q, int32_t* cu_k,
                                  int capacity, int32_t* meta, uint8_t* seg_is_pad, int skip_pad, int* status,
                                  cudaStream_t st);
cudaError_t launch_pad_fixup(void* out, float* lse, const int32_t* qids, int B, int Lq, int Hq, int Dv,
                             int64_t o_sb, int64_t o_ss, int64_t o_sh, int64_t l_sb, int64_t l_sh, cudaStream_t st);
cudaError_t launch_lse_merge(const void* o1, const float* l1, const void* o2, const float* l2, float* of, void* ob,
                             float* l, int T, int H, int D, int f16, cudaStream_t st);
// Cross-chunk segments (3 per row) of the shard [q0, q0 + Lq) against the
// earlier key chunk [k0, k0 + Lk); dev_meta = {3 B, max_q, max_k}.
cudaError_t launch_cross_segments(const int32_t* ids, int B, int S, int q0, int Lq, int k0, int Lk, int32_t* cu_q,
                                  int32_t* cu_k, int32_t* dev_meta, cudaStream_t st);
// Live-row merge and gradient add over the query rows of segments with keys
// (segment count from dev_meta when given, capped at nseg).
cudaError_t launch_lse_merge_live(float* o_acc, void* o_run, float* l_acc, const void* o_new, const float* l_new,
                                  const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta, int nseg, int T,
                                  int H, int D, int f16, cudaStream_t st);
cudaError_t launch_grad_add_live(void* dst, const void* src, const int32_t* cu_q, const int32_t* cu_k,
                                 const int32_t* dev_meta, int nseg, int T, int H, int D, int f16, cudaStream_t st);
// dQ = scale * dQacc (q's dtype and layout); with a schedule (sc), dK = scale *
// the sum of each cut key tile's partial-sum slots and dV = the sum of its
// slots (pk / pv: [slot][Hkv][128][D] fp32) for the tile's key rows.
cudaError_t launch_bwd_convert(const float* dq_acc, void* dq, bool have_q, int B, int Sq, int Hq, int Dqk,
                               int64_t q_sb, int64_t q_ss, int64_t q_sh, const SegInfo& g, const BwdSchedule* sc,
                               const float* pk, const float* pv, void* dk, void* dv, int Hkv, int Dv, int64_t k_sb,
                               int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss, int64_t v_sh, float scale,
                               int f16, cudaStream_t st);

// One CTA whose warp 0 makes one bounded pipeline wait; it runs out (and
// records kStatusTimeout in *status) unless `arrive` is set.
cudaError_t launch_wait_check(int arrive, uint64_t limit_ns, int* status, cudaStream_t st);

}  // namespace psf
