// bwd.cu -- one ring step of the backward pass on tcgen05 tensor cores.
//
// Key/value-stationary: one CTA owns a 128-row K/V tile of one key/value head
// (the shard that travels around the ring) and loops over the query heads of
// its GQA group and the 128-row query tiles of the query shard that holds this
// K/V shard at this ring step.  From the saved LSE it recomputes
//   S^T = K Q^T,  P^T = exp(scale S^T - LSE),  dP^T = V dO^T,
//   dS^T = scale P^T (dP^T - Delta),
//   dV += P^T dO,  dK += dS^T Q,  dQ += dS K,
// keeping dV and dK in tensor memory for the whole CTA and adding dQ into an
// fp32 accumulator with TMA bulk tensor reductions.
//
// Warp roles (512 threads):
//   warp 0       producer: K, V once; then Q_i with its LSE/Delta slices into a
//                ring of kNQ stages and dO_i into a ring of kNDO (2 and 1 at
//                head_dim 128, 4 and 2 at head_dim 64)
//   warp 1       TMEM owner + single-thread UMMA issuer, per pair i:
//                  [P_i written] dV_i, S_{i+1} | [dS_i written] dQ_i, dK_i |
//                  [dQ_i read out] dP_{i+1}
//                so the tensor pipe runs dV_i/S_{i+1} while the compute
//                warpgroups work on dS_i, and dQ_i/dK_i while they work on P_{i+1}
//   warps 4-11   two compute warpgroups, each on half of the 128 query columns
//                (P^T, dS^T) and, at the end, half of the head dimension of dK/dV
//   warps 12-15  dQ warpgroup: reads dQ_i out of tensor memory, stages it in its
//                own shared-memory buffer and adds it into the accumulator with
//                bulk reductions, off the compute warpgroups' path; every kChain
//                pairs it also moves the dV/dK chain into the fp32 accumulators
// Tensor memory: dV [0,D), dK [D,2D), S^T/P^T [2D,2D+128), dP^T/dQ after.
// P^T (bf16, two per column) overwrites columns [0,32) and [64,96) of S^T
// (each warpgroup packs into its own columns) and feeds the dV MMA from tensor
// memory.  dS^T goes to shared memory only (128 rows of key x 128 query
// columns, two 64-column chunks, 128-byte swizzle): the same bytes are the
// K-major A operand of dK = dS^T Q and the MN-major A operand of dQ = dS K.
#include "ring_attn_internal.h"
#include "tc.cuh"
#include "bwd_tiles.cuh"

namespace ra {
namespace {

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;   // one 128-row bf16 tile
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  // Q (with its LSE/Delta slices) and dO rings: at head_dim 64 a pair is
  // shorter than a tile's load latency, and 16 KB tiles leave room for more
  // stages
  static constexpr int kNQ = D == 64 ? 4 : 2;
  static constexpr int kNDO = D == 64 ? 2 : 1;
  static constexpr int kQ0 = 2 * kTile;                 // Q stages
  static constexpr int kDO = kQ0 + kNQ * kTile;         // dO stages
  static constexpr int kDS = kDO + kNDO * kTile;        // dS^T, 128 x 128 bf16
  static constexpr int kStg = kDS + 32768;              // dQ staging, 128 rows x 64 fp32
  static constexpr int kStat = kStg + 32768;            // per Q stage: lse2[128], delta[128]
  static constexpr int kBar = kStat + kNQ * 1024;
  static constexpr int kSmem = kBar + 256;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, false, true);   // dV, dK: A tmem, B MN-major
  static constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, true, true);    // dQ: A, B MN-major
  static constexpr uint32_t tdV = 0, tdK = D, tS = 2 * D, tP = 2 * D + 128;
  // dV/dK are accumulated in tensor memory over at most kChain pairs, then
  // added into the fp32 accumulators.  The tensor core's fp32 accumulation
  // drifts roughly in proportion to the chain length (4096 pairs: 6.6e-4
  // relative on the first keys of a 128K document); 256 pairs bound it near
  // 4e-5 and cover every CTA of a 16-step 128K ring without a flush.
  static constexpr int kChain = 256;
};

template <int D>
__global__ void __launch_bounds__(512, 1)
    ring_bwd_step_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                         const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (*reinterpret_cast<volatile int*>(p.status) != 0) return;
  if ((smem_u32(smem) & 1023u) != 0) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0) atomicCAS(p.status, 0, 299);
    return;
  }
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::kK, sV = s0 + C::kV, sQ = s0 + C::kQ0, sDO = s0 + C::kDO, sDS = s0 + C::kDS;
  const uint32_t sStg = s0 + C::kStg;
  float* stat = reinterpret_cast<float*>(smem + C::kStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  const uint32_t b_kv = smem_u32(bars + 0);
  const uint32_t b_qfull = smem_u32(bars + 17);                          // [kNQ] Q_i + LSE/Delta landed
  const uint32_t b_qempty = smem_u32(bars + 17 + C::kNQ);               // [kNQ] Q stage released (after dK_i)
  const uint32_t b_dofull = smem_u32(bars + 17 + 2 * C::kNQ);           // [kNDO] dO_i landed
  const uint32_t b_doempty = smem_u32(bars + 17 + 2 * C::kNQ + C::kNDO); // [kNDO] dO released (after dV_i)
  const uint32_t b_s = smem_u32(bars + 7);       // S^T_i in TMEM
  const uint32_t b_dp = smem_u32(bars + 8);      // dP^T_i in TMEM
  const uint32_t b_pr = smem_u32(bars + 9);      // dS^T_i written to shared memory
  const uint32_t b_dq = smem_u32(bars + 10);     // dQ_i in TMEM (and all earlier MMAs done)
  const uint32_t b_dqf = smem_u32(bars + 11);    // dQ_i read out
  const uint32_t b_drain = smem_u32(bars + 12);
  const uint32_t b_kvf = smem_u32(bars + 13);    // a finished dV/dK chain left tensor memory
  const uint32_t b_p = smem_u32(bars + 14);      // P^T_i packed in tensor memory
  const uint32_t b_dsf = smem_u32(bars + 15);    // dQ_i and dK_i done: the dS buffer may be rewritten
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdItem it = p.items[blockIdx.x];
  const int g = it.flags >> kHeadShift;
  PairList pl;
  pl.qb0 = it.qb0; pl.qe0 = it.qe0; pl.qb1 = it.qb1; pl.qe1 = it.qe1;
  pl.n0 = ceil128(it.qb0 & ~3, it.qe0);
  pl.nt = pl.n0 + ceil128(it.qb1 & ~3, it.qe1);
  pl.G = p.Hq / p.Hkv;
  pl.hbase = g * pl.G;
  const int npairs = pl.nt * pl.G;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int x = 0; x < C::kNQ; ++x) { mbar_init(b_qfull + 8 * x, 1); mbar_init(b_qempty + 8 * x, 1); }
    for (int x = 0; x < C::kNDO; ++x) { mbar_init(b_dofull + 8 * x, 1); mbar_init(b_doempty + 8 * x, 1); }
    mbar_init(b_s, 1); mbar_init(b_dp, 1);
    mbar_init(b_pr, 8);    // arrivals are one per warp (8 compute warps): the shared-memory
                           // unit takes an mbarrier's arrivals one at a time
    mbar_init(b_dq, 1);
    mbar_init(b_dqf, 4);
    mbar_init(b_drain, 1);
    mbar_init(b_kvf, 4);
    mbar_init(b_p, 8);
    mbar_init(b_dsf, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.status};
  // all lanes of a warp take the same branch after a bounded wait
  auto wait_warp = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, site)) != 0;
  };

  // Register split: 512 threads x 128 at launch = 65536.  Producer/MMA
  // warpgroup 80, compute warpgroups 168, dQ warpgroup 88:
  // 128 x 80 + 256 x 168 + 128 x 88 = 64512.  Each warpgroup sets its limit at
  // the head of its own branch.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      bool ok = true;
      int issued_q = 0, issued_do = 0;
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmL); tma_prefetch_desc(&tmD);
      mbar_expect_tx(b_kv, 2 * C::kTile);
      for (int hf = 0; hf < D / 64; ++hf) {
        tma_load_3d(sK + hf * 16384, &tmK, b_kv, 64 * hf, g, it.k0);
        tma_load_3d(sV + hf * 16384, &tmV, b_kv, 64 * hf, g, it.k0);
      }
      for (int i = 0; i < npairs; ++i) {
        const int st = i % C::kNQ, sd = i % C::kNDO;
        const int h = pl.head(i), q0 = pl.start(i);
        if (!mbar_wait(b_qempty + 8 * st, ((i / C::kNQ) & 1) ^ 1, ab, 201)) { ok = false; break; }
        const uint32_t sq = sQ + st * C::kTile;
        const uint32_t sl = smem_u32(stat + st * 256);
        mbar_expect_tx(b_qfull + 8 * st, C::kTile + 2 * 512);
        for (int hf = 0; hf < D / 64; ++hf) tma_load_3d(sq + hf * 16384, &tmQ, b_qfull + 8 * st, 64 * hf, h, q0);
        // LSE (log2 units) and Delta of the tile's 128 query columns
        tma_load_2d(sl, &tmL, b_qfull + 8 * st, q0, h);
        tma_load_2d(sl + 512, &tmD, b_qfull + 8 * st, q0, h);
        ++issued_q;
        if (!mbar_wait(b_doempty + 8 * sd, ((i / C::kNDO) & 1) ^ 1, ab, 206)) { ok = false; break; }
        mbar_expect_tx(b_dofull + 8 * sd, C::kTile);
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_3d(sDO + sd * C::kTile + hf * 16384, &tmDO, b_dofull + 8 * sd, 64 * hf, h, q0);
        ++issued_do;
      }
      {
        // CTAs run one per SM and start in order, so CTA b + next_cta takes an
        // SM about when this one ends: bring its K/V tile into L2 now.
        const long long nb = (long long)blockIdx.x + p.next_cta;
        if (ok && p.next_cta > 0 && nb < (long long)gridDim.x) {
          const BwdItem nx = p.items[nb];
          const int ng = nx.flags >> kHeadShift;
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_prefetch_l2_3d(&tmK, 64 * hf, ng, nx.k0);
            tma_prefetch_l2_3d(&tmV, 64 * hf, ng, nx.k0);
          }
        }
      }
      if (!ok) {  // drain this CTA's copies still in flight
        mbar_wait_drain(b_kv, 0);
        for (int i = issued_q > C::kNQ ? issued_q - C::kNQ : 0; i < issued_q; ++i)
          mbar_wait_drain(b_qfull + 8 * (i % C::kNQ), (i / C::kNQ) & 1);
        for (int i = issued_do > C::kNDO ? issued_do - C::kNDO : 0; i < issued_do; ++i)
          mbar_wait_drain(b_dofull + 8 * (i % C::kNDO), (i / C::kNDO) & 1);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // Every operand descriptor is the shared-memory base's plus constants
      // (sdesc_at): each MMA costs two adds to issue, so the single issuing
      // thread keeps up with the tensor pipe.  K-major operands: lbo 16;
      // MN-major: lbo = the 64-column block stride.
      const uint64_t d0 = sdesc_sw128(s0, 0, 1024);
      auto issue_s = [&](int i) {  // S^T_i = K Q_i^T
        const uint64_t dk = opaque(d0);
        const uint64_t dq = sdesc_at(dk, (uint32_t)(i % C::kNQ) * C::kTile, 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tmem + C::tS, sdesc_at(dk, C::kK + off, 16), sdesc_at(dq, C::kQ0 + off, 16), C::kIdescS, kk > 0);
        }
        umma_commit(b_s);
      };
      auto issue_dp = [&](int i) {  // dP^T_i = V dO_i^T
        const uint64_t dv = opaque(d0);
        const uint64_t dd = sdesc_at(dv, (uint32_t)(i % C::kNDO) * C::kTile, 0);  // dO_i's stage
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tmem + C::tP, sdesc_at(dv, C::kV + off, 16), sdesc_at(dd, C::kDO + off, 16), C::kIdescS, kk > 0);
        }
        umma_commit(b_dp);
      };
      bool ok = mbar_wait(b_kv, 0, ab, 202);
      if (ok && npairs > 0) {
        ok = mbar_wait(b_qfull, 0, ab, 203) && mbar_wait(b_dofull, 0, ab, 207);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
      }
      for (int i = 0; i < npairs && ok; ++i) {
        const int st = i % C::kNQ, sd = i % C::kNDO;
        const uint32_t pi = i & 1;
        const uint64_t db = opaque(d0);
        const uint64_t dq = sdesc_at(db, (uint32_t)st * C::kTile, 0);  // this pair's Q stage
        const uint64_t dd = sdesc_at(db, (uint32_t)sd * C::kTile, 0);  // this pair's dO stage
        // dV += P^T dO once P_i is packed (A from tensor memory: query columns
        // 0-63 in columns [0,32) of the S region, 64-127 in [64,96); B MN-major)
        if (!mbar_wait(b_p, pi, ab, 205)) { ok = false; break; }
        if (i > 0 && i % C::kChain == 0) {  // the previous dV/dK chain has been flushed
          if (!mbar_wait(b_kvf, ((i / C::kChain) - 1) & 1, ab, 208)) { ok = false; break; }
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + C::tdV, tmem + C::tS + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_at(dd, C::kDO + kk * 2048, 16384),
                  C::kIdescG, (i % C::kChain > 0 || kk > 0) ? 1u : 0u);
        umma_commit(b_doempty + 8 * sd);
        // S_{i+1} right behind dV_i, the last reader of P_i in the S region
        if (i + 1 < npairs) {
          if (!mbar_wait(b_qfull + 8 * ((i + 1) % C::kNQ), ((i + 1) / C::kNQ) & 1, ab, 203)) { ok = false; break; }
          tc_fence_after();
          issue_s(i + 1);
        }
        // dQ_i = dS K and dK += dS^T Q, once dS_i is in shared memory (and the
        // compute warpgroups have read dP_i, whose region dQ_i takes)
        if (!mbar_wait(b_pr, pi, ab, 206)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + C::tP, sdesc_at(db, C::kDS + kk * 2048, 16384), sdesc_at(db, C::kK + kk * 2048, 16384),
                  C::kIdescQ, kk > 0);
        umma_commit(b_dq);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + C::tdK, sdesc_at(db, C::kDS + (kk >> 2) * 16384 + (kk & 3) * 32, 16),
                  sdesc_at(dq, C::kQ0 + kk * 2048, 16384), C::kIdescG, (i % C::kChain > 0 || kk > 0) ? 1u : 0u);
        umma_commit(b_qempty + 8 * st);
        umma_commit(b_dsf);
        // dP_{i+1} once dQ_i has left the region and dO_{i+1} has landed
        if (i + 1 < npairs) {
          if (!mbar_wait(b_dqf, pi, ab, 204)) { ok = false; break; }
          if (!mbar_wait(b_dofull + 8 * ((i + 1) % C::kNDO), ((i + 1) / C::kNDO) & 1, ab, 207)) { ok = false; break; }
          tc_fence_after();
          issue_dp(i + 1);
        }
      }
      if (!ok) {  // let issued MMAs finish before tensor memory is released
        umma_commit(b_drain);
        mbar_wait_drain(b_drain, 0);
      }
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;");
    // ------------------------------------------------------------ compute warpgroups
    // Two warpgroups split every 128-column tile: warpgroup w takes query
    // columns [64w, 64w + 64) of S^T/dP^T, and head-dim columns [D/2 w, D/2 (w+1))
    // of the final dK and dV.  TMEM lanes = key rows.
    const int wg = (warp - 4) >> 2;
    const int tid = threadIdx.x - 128 * (1 + wg);
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t tS = tmem_addr(tmem, lane_base, C::tS);
    const uint32_t tP = tmem_addr(tmem, lane_base, C::tP);
    const int krow = it.k0 + tid;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2), scale2 = f2_pack(p.scale, p.scale);
    constexpr int DH = D / 2;  // head-dim columns per warpgroup
    const uint32_t row_addr = sDS + wg * 16384 + tid * 128;
    // add this warpgroup's half of dV and dK (tensor memory, lanes = key rows)
    // into the fp32 accumulators
    const bool valid = krow < it.k1;
    float* dv_row = p.dv_acc + ((size_t)krow * p.Hkv + g) * D + wg * DH;
    float* dk_row = p.dk_acc + ((size_t)krow * p.Hkv + g) * D + wg * DH;
    auto flush_dkdv = [&]() {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t t = tmem_addr(tmem, lane_base, (which == 0 ? C::tdV : C::tdK) + wg * DH);
        float* dst = which == 0 ? dv_row : dk_row;
#pragma unroll
        for (int c = 0; c < DH / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(t + 32 * c, r);
          tmem_ld_wait();
          reg_fence32(r);
          if (valid) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
              red_add_v4(dst + 32 * c + 4 * x, __uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                         __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
      }
    };
    // visible query columns c of pair i satisfy  qlo <= q0 + c < qe  and
    // (causal) krow <= q0 + c
    auto vis = [&](int i, bool& need_mask, int& cmin, int& cmax) {
      const int q0 = pl.start(i), qlo = pl.lo(i), qe = pl.end(i);
      need_mask = (it.k1 - it.k0 < 128) || (q0 + 128 > qe) || (q0 < qlo) || (p.causal && it.k1 - 1 > q0);
      cmin = (krow >= it.k1) ? 128 : max(qlo - q0, p.causal ? krow - q0 : 0);
      cmax = qe - q0;  // exclusive
    };
    // P^T of the current pair times the softmax scale, as packed fp32 pairs
    // (masked), kept for its dS phase: dS is formed from the unrounded P, so
    // it carries one bf16 rounding (its own, for the dK/dQ MMAs) instead of
    // two; only the dV MMA consumes the bf16-rounded P.
    uint64_t pf[32];
    // ---- P^T = exp2(S^T scale log2e - LSE log2e) on columns [64 wg, 64 wg + 64),
    // packed into this warpgroup's own columns of the S region (never into the
    // other warpgroup's columns, which it may not have read yet)
    auto p_phase = [&](int i) -> bool {
      if (!wait_warp(b_s, i & 1, 210)) return false;
      tc_fence_after();
      bool need_mask;
      int cmin, cmax;
      vis(i, need_mask, cmin, cmax);
      const float4* sl4 = reinterpret_cast<const float4*>(stat + (i % C::kNQ) * 256);
      uint32_t r[2][32];
      tmem_ld32(tS + 64 * wg, r[0]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      tmem_ld32(tS + 64 * wg + 32, r[1]);  // in flight while the first 32 columns are computed
      uint32_t w0[16], w1[16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c == 1) {
          tmem_ld_wait();
          reg_fence32(r[1]);
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = 64 * wg + 32 * c + 2 * x;
          const float4 l4 = sl4[c0 >> 2];  // broadcast read of 4 columns' -LSE log2e
          const uint64_t nl = (x & 1) ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y);
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][2 * x]), __uint_as_float(r[c][2 * x + 1])), sl2x2, nl), x0,
                    x1);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (need_mask) {
            if (c0 < cmin || c0 >= cmax) p0 = 0.f;
            if (c0 + 1 < cmin || c0 + 1 >= cmax) p1 = 0.f;
          }
          pf[16 * c + x] = f2_mul(f2_pack(p0, p1), scale2);
          (c == 0 ? w0 : w1)[x] = pack_bf16x2(p0, p1);
        }
      }
      tmem_st16(tS + 64 * wg, w0);
      tmem_st16(tS + 64 * wg + 16, w1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p);
      return true;
    };
    // ---- dS^T = scale P^T (dP^T - Delta), to shared memory (this warpgroup's
    // 64 query columns are chunk `wg`) once dQ_{i-1} and dK_{i-1} have read the
    // previous one
    auto ds_phase = [&](int i) -> bool {
      if (!wait_warp(b_dp, i & 1, 211)) return false;
      tc_fence_after();
      const float4* sl4 = reinterpret_cast<const float4*>(stat + (i % C::kNQ) * 256);
      uint32_t r[2][32];
      tmem_ld32(tP + 64 * wg, r[0]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      tmem_ld32(tP + 64 * wg + 32, r[1]);  // in flight while the first 32 columns are computed
      uint32_t w[2][16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c == 1) {
          tmem_ld_wait();
          reg_fence32(r[1]);
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = 64 * wg + 32 * c + 2 * x;
          const float4 d4 = sl4[32 + (c0 >> 2)];  // broadcast read of 4 columns' -Delta
          const uint64_t nd = (x & 1) ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
          float d0, d1;  // scale P (dP - Delta)
          f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(r[c][2 * x]), __uint_as_float(r[c][2 * x + 1])), nd),
                           pf[16 * c + x]),
                    d0, d1);
          w[c][x] = pack_bf16x2(d0, d1);
        }
      }
      // dP_i is in registers: its tensor-memory region may take dQ_i
      tc_fence_before();
      if (i > 0 && !wait_warp(b_dsf, (i - 1) & 1, 212)) return false;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const int piece = c * 4 + pc;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row_addr + ((piece ^ (tid & 7)) << 4)),
                       "r"(w[c][4 * pc]), "r"(w[c][4 * pc + 1]), "r"(w[c][4 * pc + 2]), "r"(w[c][4 * pc + 3])
                       : "memory");
        }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pr);
      return true;
    };
    bool ok = npairs == 0 || p_phase(0);
    for (int i = 0; i < npairs && ok; ++i) {
      ok = ds_phase(i);
      if (ok && i + 1 < npairs) ok = p_phase(i + 1);
    }
    // every MMA of the CTA is done once dQ and dK of the last pair are
    if (ok && npairs > 0 && wait_warp(b_dsf, (npairs - 1) & 1, 213)) {
      tc_fence_after();
      flush_dkdv();
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
    // ------------------------------------------------------------ dQ warpgroup
    // TMEM lanes = query rows.  For every pair: read dQ_i (64 columns at a
    // time), stage it in this warpgroup's buffer (each warp its own 32 rows,
    // two 32-column boxes per 64 columns, 128-byte swizzle) and add it into the
    // fp32 accumulator with bulk tensor reductions.  Rows outside the query
    // range carry exact zeros (their dS columns are masked); rows past T are
    // clipped by the tensor map.
    const int tid = threadIdx.x - 384;
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t tQ = tmem_addr(tmem, lane_base, C::tP);
    const uint32_t wbuf = sStg + (uint32_t)(warp & 3) * 8192;  // this warp's 8 KB
    const uint32_t row = (uint32_t)lane * 128;
    const bool lead = lane == 0;
    for (int j = 0; j < npairs; ++j) {
      if (!wait_warp(b_dq, j & 1, 220)) break;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        uint32_t r[2][32];
        tmem_ld32(tQ + 64 * half, r[0]);
        tmem_ld32(tQ + 64 * half + 32, r[1]);
        tmem_ld_wait();
        reg_fence32(r[0]);
        reg_fence32(r[1]);
        if (half == D / 64 - 1) {  // all of dQ_j is in registers or staged: release tensor memory
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_dqf);
        }
        if (lead) bulk_wait_read();  // the buffer's previous boxes have been read
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int pc = 0; pc < 8; ++pc)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(wbuf + k * 4096 + row +
                                                                          ((pc ^ (lane & 7)) << 4)),
                         "r"(r[k][4 * pc]), "r"(r[k][4 * pc + 1]), "r"(r[k][4 * pc + 2]), "r"(r[k][4 * pc + 3])
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lead) {
          tma_reduce_add_3d(&tmDQ, wbuf, 64 * half, pl.head(j), pl.start(j) + (tid & ~31));
          tma_reduce_add_3d(&tmDQ, wbuf + 4096, 64 * half + 32, pl.head(j), pl.start(j) + (tid & ~31));
          bulk_commit();
        }
      }
      // pair j closed a dV/dK chain (all of its MMAs are done: b_dq of pair j)
      // and more pairs follow: add the chain into the fp32 accumulators, so the
      // MMA can restart the chain in tensor memory.  Here lanes = key rows.
      if ((j + 1) % C::kChain == 0 && j + 1 < npairs) {
        if (!wait_warp(b_dsf, j & 1, 221)) break;  // dK_j (issued after dQ_j) is done too
        tc_fence_after();
        const int krow = it.k0 + tid;
        const bool valid = krow < it.k1;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t t = tmem_addr(tmem, lane_base, which == 0 ? C::tdV : C::tdK);
          float* dst = (which == 0 ? p.dv_acc : p.dk_acc) + ((size_t)krow * p.Hkv + g) * D;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(t + 32 * c, r);
            tmem_ld_wait();
            reg_fence32(r);
            if (valid) {
#pragma unroll
              for (int x = 0; x < 8; ++x)
                red_add_v4(dst + 32 * c + 4 * x, __uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                           __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_kvf);
      }
    }
    if (lead) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                   const CUtensorMap& tl, const CUtensorMap& td, const CUtensorMap& tdq, const BwdParams& p,
                   int num_items, cudaStream_t stream) {
  auto kern = ring_bwd_step_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)num_items;
  if (grid <= 0) return cudaSuccess;
  BwdParams q = p;  // one CTA per SM (shared memory): the stride to the CTA that follows on an SM
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  q.next_cta = sms;
  // (Overlapping consecutive backward ring steps, as the forward does, was
  // measured slower: two query shards' dQ rows then share L2.)
  kern<<<(unsigned)grid, 512, BwdCfg<D>::kSmem, stream>>>(tq, tk, tv, tdo, tl, td, tdq, q);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_step(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tl, const CUtensorMap& td,
                            const CUtensorMap& tdq, const BwdParams& p, int num_items, cudaStream_t stream) {
  if (head_dim == 128) return launch<128>(tq, tk, tv, tdo, tl, td, tdq, p, num_items, stream);
  if (head_dim == 64) return launch<64>(tq, tk, tv, tdo, tl, td, tdq, p, num_items, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ra
