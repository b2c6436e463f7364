// ring_attn_internal.h -- work-item layouts shared by the host planner and the
// kernels, and the kernel launch wrappers.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/ring_attn.h"

namespace ra {

// Forward work item: one CTA = up to 256 query rows (two 128-row tiles; one
// tile at head_dim 256) of one query chunk, all in one document, against up to two key ranges of the
// key/value shard that the query shard holds at this ring step.  Ranges are
// global token positions, sorted, disjoint, already clipped to the keys the
// rows may see (for causal: keys < q1).  Grid: items x Hq.
struct FwdItem {
  int32_t q0, q1;    // query rows [q0, q1), q1 - q0 <= 256
  int32_t kb0, ke0;  // key range 0 (may be empty)
  int32_t kb1, ke1;  // key range 1 (may be empty)
  int32_t flags;     // kFirstStep: write the running state instead of merging
  int32_t tiles;     // number of 128-key tiles (work estimate)
};

// Backward work item: one CTA = one 128-row key/value tile of one key/value
// head (flags >> kHeadShift), against up to two query ranges of the query
// shard that holds this key/value shard at this ring step (for causal:
// queries >= k0).  The CTA loops over the Hq/Hkv query heads of the group.
// Grid: one CTA per item.
struct BwdItem {
  int32_t k0, k1;    // key rows [k0, k1), k1 - k0 <= 128
  int32_t qb0, qe0;  // query range 0 (may be empty)
  int32_t qb1, qe1;  // query range 1 (may be empty)
  int32_t flags;
  int32_t tiles;     // number of 128-query tiles (work estimate)
};

constexpr int32_t kFirstStep = 1;
constexpr int32_t kHeadShift = 8;  // backward items: key/value head in flags bits [8, 31)

struct FwdParams {
  const FwdItem* items;
  int32_t Hq, Hkv, T, causal;
  float scale_log2;  // softmax scale * log2(e)
  float* o_run;      // fp32 [T, Hq, D] running (normalised) output (ring-step launches)
  float* lse;        // fp32 [Hq, T] running log-sum-exp (natural log)
  int* status;       // workspace status word
  int32_t next_cta;  // ring-step launches: CTAs resident at once (one per SM)
  // single launch over all ring steps: per-tile (start, range end) table and
  // the final output, written once (bf16 or fp32)
  const int2* tiles;
  void* o_out;
  int32_t o_bf16;
};

struct BwdParams {
  const BwdItem* items;
  int32_t Hq, Hkv, T, causal;
  float scale_log2;    // softmax scale * log2(e)
  float scale;         // softmax scale
  const float* lse2;   // [Hq, stat_pitch] LSE * log2(e)
  const float* delta;  // [Hq, stat_pitch] -rowsum(dO * O), times the softmax scale at head_dim 256
  int64_t stat_pitch;  // T rounded up to a multiple of 4
  float* dq_acc;       // fp32 [T, Hq, D], scaled dq accumulated with bulk reductions
  float* dk_acc;       // fp32 [T, Hkv, D]
  float* dv_acc;       // fp32 [T, Hkv, D]
  int* status;
  int32_t next_cta;    // CTAs resident at once (one per SM)
};

// Record `msg` as this thread's last error text and return `st`.
ra_status set_last_error(ra_status st, const char* msg);

// Kernel launch wrappers (return the launch error).
cudaError_t launch_fwd_fused(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int num_items, cudaStream_t stream);
cudaError_t launch_fwd_step(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const FwdParams& p, int num_items,
                            cudaStream_t stream);
// head_dim 256 (fwd256.cu): one 128-row query tile per CTA
cudaError_t launch_fwd_step_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const FwdParams& p, int num_items, cudaStream_t stream);
cudaError_t launch_fwd_fused_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const FwdParams& p, int num_items, cudaStream_t stream);
// head_dim 128 (bwd_pair.cu): clusters of two CTAs over two key tiles; the
// items come in pairs (num_items even), q64/dout64 with 64-row boxes.
cudaError_t launch_bwd_step_pair(const CUtensorMap& tq, const CUtensorMap& tq64, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdo64,
                                 const CUtensorMap& tl, const CUtensorMap& td, const CUtensorMap& tdq,
                                 const BwdParams& p, int num_items, cudaStream_t stream);
cudaError_t launch_bwd_step(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tlse2,
                            const CUtensorMap& tdelta, const CUtensorMap& tdq_acc, const BwdParams& p,
                            int num_items, cudaStream_t stream);
// head_dim 256 (bwd256.cu): two CTAs per work item (column halves), 64-row query tiles
cudaError_t launch_bwd_step_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tl, const CUtensorMap& td,
                                 const CUtensorMap& tdq, const BwdParams& p, int num_items, cudaStream_t stream);
// o (bf16) = o_run (fp32), elementwise.
cudaError_t launch_cast_bf16(const float* src, void* dst, size_t n, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(int* status, uint64_t limit_ns, int site, cudaStream_t stream);
// delta[h, t] = -s * sum_d dO[t,h,d] * O[t,h,d];  lse2[h, t] = -lse[h, t] * log2(e)
// (negated, as the backward's compute phases consume them; s = the softmax
// scale at head_dim 256, whose dS phase folds the scale into one fma, else 1);
// both written with row pitch `pitch` (>= T).
cudaError_t launch_bwd_preprocess(const void* o, int o_is_fp32, const void* dout, const float* lse,
                                  float* delta, float* lse2, int T, int64_t pitch, int Hq, int D, float scale,
                                  cudaStream_t stream);

}  // namespace ra
