// bwd_pair.cu -- one ring step of the backward pass at head_dim 128 on CTA
// pairs (cta_group::2 tensor cores).
//
// The same recomputation as the one-CTA kernel (bwd.cu), from the saved LSE:
//   S^T = K Q^T,  P^T = exp(scale S^T - LSE),  dP^T = V dO^T,
//   dS^T = scale P^T (dP^T - Delta),
//   dV += P^T dO,  dK += dS^T Q,  dQ += dS K,
// but a cluster of two CTAs takes two neighbouring 128-row key tiles of one
// key/value head (CTA r: tile r) and walks the same query tiles.  The even CTA
// issues every MMA for both:
//   S^T, dP^T  M = 256 (the pair's 256 keys), N = 128 queries: CTA r supplies
//              query rows [64r, 64r + 64) of Q (dO), all 128 columns;
//   dV, dK     M = 256 keys, N = 128 head columns, A (P^T, dS^T) from each
//              CTA's tensor memory: CTA r supplies head columns [64r, 64r + 64)
//              of dO (Q) for all 128 query rows;
//   dQ         M = 128 queries, N = 128 head columns, reduced over all 256
//              keys: CTA r supplies dS of query rows [64r, 64r + 64) for both
//              key tiles and head columns [64r, 64r + 64) of K for both key
//              tiles, and receives dQ of its 64 query rows (all columns).
// So each B operand is read half from each CTA's shared memory, and the pair
// adds dQ of 256 keys into the accumulator once.  Each CTA loads its own tiles
// (no multicast).  dS^T of the other CTA's query rows goes to the other CTA's
// shared memory with cluster stores; the K columns dQ needs from the other key
// tile are loaded once.
//
// Warp roles (512 threads in each CTA):
//   warp 0       producer: its own tiles; loads complete on the even CTA's
//                barriers (the MMA issuer's), the even CTA's producer posting
//                both CTAs' byte counts
//   warp 1       tensor memory (both CTAs); in the even CTA the MMA issuer:
//                  [P_i written] dV_i, S_{i+1} | [dS_i written] dQ_i, dK_i |
//                  [dQ_i read out] dP_{i+1}
//   warps 4-11   two compute warpgroups on the CTA's 128 keys (TMEM lanes),
//                each on 64 query columns: P^T, dS^T (into tensor memory for dK
//                and into shared memory of the CTA whose query rows they are,
//                for dQ); at the end half of the head columns of dK/dV each
//   warps 12-15  dQ warpgroup: reads the CTA's dQ rows out of tensor memory,
//                stages and adds them with bulk tensor reductions; every kChain
//                pairs it moves the dV/dK chain into the fp32 accumulators
// Tensor memory (each CTA): dV [0,128), dK [128,256), S^T/P^T [256,384),
// dP^T [384,512).  P^T (bf16, two per column) overwrites columns [0,32) and
// [64,96) of the S^T region; dS^T (bf16) overwrites columns [0,32) and
// [96,128) of the dP^T region, and dQ takes its columns [32,96): dQ and dK
// of a pair do not share columns, so dQ runs first and its read-out overlaps dK.
#include "ring_attn_internal.h"
#include "tc.cuh"
#include "bwd_tiles.cuh"

namespace ra {
namespace {

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kK = 0;          // own K tile: 128 keys x 128 columns, two 64-column boxes
  static constexpr int kV = 32768;      // own V tile
  static constexpr int kKB = 65536;     // [2] K of key tile t, this CTA's 64 head columns (dQ's B)
  static constexpr int kQS = 98304;     // [2 stages] this CTA's 64 query rows of Q, two 64-column boxes
  static constexpr int kQK = 131072;    // all 128 query rows of Q, this CTA's 64 head columns (dK's B)
  static constexpr int kDOP = 147456;   // this CTA's 64 query rows of dO, two boxes (dP's B)
  static constexpr int kDOV = 163840;   // all 128 query rows of dO, this CTA's 64 head columns (dV's B)
  static constexpr int kR = 180224;     // [2] dS^T of key tile t, this CTA's 64 query columns (dQ's A)
  static constexpr int kStg = 212992;   // dQ staging: 4 warps x 32 rows x 32 fp32
  static constexpr int kStat = 229376;  // [2 stages] -LSE log2e [128], -Delta [128]
  static constexpr int kBar = kStat + 2048;
  static constexpr int kSmem = kBar + 256;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(256, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t kIdescG = idesc_bf16_f32(256, 128, false, true);   // dV, dK: A tmem, B MN-major
  static constexpr uint32_t kIdescQ = idesc_bf16_f32(128, 128, true, true);    // dQ: A, B MN-major
  static constexpr uint32_t tdV = 0, tdK = 128, tS = 256, tP = 384, tQ = 416;
  // dV/dK accumulate in tensor memory over at most kChain pairs between flushes
  // (as in the one-CTA kernel).
  static constexpr int kChain = 256;
};
static_assert(PairCfg::kSmem <= 232448, "shared memory of one CTA");

__global__ void __launch_bounds__(512, 1)
    ring_bwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQ64,
                         const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmDO64,
                         const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                         const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = PairCfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s0 = smem_u32(smem);
  float* stat = reinterpret_cast<float*>(smem + C::kStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  const uint32_t b_kv = smem_u32(bars + 0);       // K, V, KB landed (both CTAs; even CTA)
  const uint32_t b_qsfull = smem_u32(bars + 1);   // [2] Q rows + LSE/Delta landed (even CTA)
  const uint32_t b_qsempty = smem_u32(bars + 3);  // [2] Q-row stage free (after dK_i)
  const uint32_t b_qkfull = smem_u32(bars + 5);   // Q columns landed (even CTA)
  const uint32_t b_qkempty = smem_u32(bars + 6);  // after dK_i
  const uint32_t b_dopfull = smem_u32(bars + 7);  // dO rows landed (even CTA)
  const uint32_t b_dopempty = smem_u32(bars + 8); // after dP_i
  const uint32_t b_dovfull = smem_u32(bars + 9);  // dO columns landed (even CTA)
  const uint32_t b_dovempty = smem_u32(bars + 10);// after dV_i
  const uint32_t b_s = smem_u32(bars + 11);       // S^T_i in tensor memory
  const uint32_t b_dp = smem_u32(bars + 12);      // dP^T_i in tensor memory
  const uint32_t b_dq = smem_u32(bars + 13);      // dQ_i in tensor memory (and all earlier MMAs done)
  const uint32_t b_dsf = smem_u32(bars + 14);     // dQ_i and dK_i done: dS buffers may be rewritten
  const uint32_t b_p = smem_u32(bars + 15);       // P^T_i packed (16 compute warps of the pair; even CTA)
  const uint32_t b_pr = smem_u32(bars + 16);      // dS^T_i written (16 compute warps; even CTA)
  const uint32_t b_dqf = smem_u32(bars + 17);     // dQ_i read out (8 dQ warps; even CTA)
  const uint32_t b_kvf = smem_u32(bars + 18);     // a dV/dK chain left tensor memory (8 warps; even CTA)
  const uint32_t b_drain = smem_u32(bars + 19);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* skip = abort_flag + 1;  // [3] entry status seen by CTA 0, CTA 1; either

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const BwdItem it = p.items[blockIdx.x];
  const int pk0 = p.items[blockIdx.x & ~1u].k0, pk1 = p.items[blockIdx.x | 1u].k0;  // key tiles 0, 1
  const int g = it.flags >> kHeadShift;
  PairList pl;
  pl.qb0 = it.qb0; pl.qe0 = it.qe0; pl.qb1 = it.qb1; pl.qe1 = it.qe1;
  pl.n0 = ceil128(it.qb0 & ~3, it.qe0);
  pl.nt = pl.n0 + ceil128(it.qb1 & ~3, it.qe1);
  pl.G = p.Hq / p.Hkv;
  pl.hbase = g * pl.G;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    mbar_init(b_qsfull, 1); mbar_init(b_qsfull + 8, 1);
    mbar_init(b_qsempty, 1); mbar_init(b_qsempty + 8, 1);
    mbar_init(b_qkfull, 1); mbar_init(b_qkempty, 1);
    mbar_init(b_dopfull, 1); mbar_init(b_dopempty, 1);
    mbar_init(b_dovfull, 1); mbar_init(b_dovempty, 1);
    mbar_init(b_s, 1); mbar_init(b_dp, 1); mbar_init(b_dq, 1); mbar_init(b_dsf, 1);
    mbar_init(b_p, 16); mbar_init(b_pr, 16);   // one arrival per compute warp of the pair
    mbar_init(b_dqf, 8); mbar_init(b_kvf, 8);  // one per dQ warp of the pair
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    // the status word as this CTA sees it (the pair must take one path: the
    // other CTA reads this after the cluster barrier below)
    skip[rank] = (*reinterpret_cast<volatile int*>(p.status) != 0 || (s0 & 1023u) != 0) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    uint32_t other;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(other) : "r"(mapa_shared(smem_u32(skip + (rank ^ 1u)), rank ^ 1u))
                 : "memory");
    skip[2] = skip[rank] | (int)other;
    if ((s0 & 1023u) != 0) atomicCAS(p.status, 0, 299);  // the 128-byte swizzle needs 1024-byte aligned tiles
  }
  __syncthreads();
  const int npairs = skip[2] ? 0 : pl.nt * pl.G;
  const Abort ab{abort_flag, p.status};
  auto wait_warp = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, ab, site)) != 0;
  };
  // the even CTA's copy of a barrier (shared::cluster address)
  auto lead = [&](uint32_t bar) { return mapa_shared(bar, 0); };
  // a handoff to the issuer: a cluster-scope release arrive on the even CTA's
  // barrier (it carries the arriving warp's writes, in either CTA)
  auto arrive_lead = [&](uint32_t bar) { mbar_arrive_cluster(lead(bar)); };

  // Register split as in the one-CTA kernel: 128 x 80 + 256 x 168 + 128 x 88 = 64512.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    if (warp == 0 && lane == 0 && npairs > 0) {
      // ---------------------------------------------------------- producer
      bool ok = true;
      int issued_qs = 0, issued_qk = 0, issued_dop = 0, issued_dov = 0;
      const uint32_t mine = 64u * rank;  // this CTA's 64 query rows / head columns
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmQ64); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO); tma_prefetch_desc(&tmDO64); tma_prefetch_desc(&tmL); tma_prefetch_desc(&tmD);
      if (even) mbar_expect_tx(b_kv, 2 * (4 * 16384 + 2 * 16384));
      for (int hf = 0; hf < 2; ++hf) {
        tma_load_3d_pair(s0 + C::kK + hf * 16384, &tmK, lead(b_kv), 64 * hf, g, it.k0);
        tma_load_3d_pair(s0 + C::kV + hf * 16384, &tmV, lead(b_kv), 64 * hf, g, it.k0);
      }
      tma_load_3d_pair(s0 + C::kKB, &tmK, lead(b_kv), (int)mine, g, pk0);
      tma_load_3d_pair(s0 + C::kKB + 16384, &tmK, lead(b_kv), (int)mine, g, pk1);
      for (int i = 0; i < npairs; ++i) {
        const int st = i & 1;
        const int h = pl.head(i), q0 = pl.start(i);
        // this CTA's query rows of Q, with the tile's LSE and Delta
        if (!mbar_wait_cluster(b_qsempty + 8 * st, ((i >> 1) & 1) ^ 1, ab, 231)) { ok = false; break; }
        if (even) mbar_expect_tx(b_qsfull + 8 * st, 2 * (16384 + 1024));
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d_pair(s0 + C::kQS + st * 16384 + hf * 8192, &tmQ64, lead(b_qsfull + 8 * st), 64 * hf, h,
                           q0 + (int)mine);
        tma_load_2d_pair(s0 + C::kStat + st * 1024, &tmL, lead(b_qsfull + 8 * st), q0, h);
        tma_load_2d_pair(s0 + C::kStat + st * 1024 + 512, &tmD, lead(b_qsfull + 8 * st), q0, h);
        ++issued_qs;
        // this CTA's query rows of dO
        if (!mbar_wait_cluster(b_dopempty, (i & 1) ^ 1, ab, 232)) { ok = false; break; }
        if (even) mbar_expect_tx(b_dopfull, 2 * 16384);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d_pair(s0 + C::kDOP + hf * 8192, &tmDO64, lead(b_dopfull), 64 * hf, h, q0 + (int)mine);
        ++issued_dop;
        // this CTA's head columns of dO and of Q, all query rows
        if (!mbar_wait_cluster(b_dovempty, (i & 1) ^ 1, ab, 233)) { ok = false; break; }
        if (even) mbar_expect_tx(b_dovfull, 2 * 16384);
        tma_load_3d_pair(s0 + C::kDOV, &tmDO, lead(b_dovfull), (int)mine, h, q0);
        ++issued_dov;
        if (!mbar_wait_cluster(b_qkempty, (i & 1) ^ 1, ab, 234)) { ok = false; break; }
        if (even) mbar_expect_tx(b_qkfull, 2 * 16384);
        tma_load_3d_pair(s0 + C::kQK, &tmQ, lead(b_qkfull), (int)mine, h, q0);
        ++issued_qk;
      }
      {
        // the K/V tile of the CTA that follows on this SM, into L2
        const long long nb = (long long)blockIdx.x + p.next_cta;
        if (ok && p.next_cta > 0 && nb < (long long)gridDim.x) {
          const BwdItem nx = p.items[nb];
          const int ng = nx.flags >> kHeadShift;
          for (int hf = 0; hf < 2; ++hf) {
            tma_prefetch_l2_3d(&tmK, 64 * hf, ng, nx.k0);
            tma_prefetch_l2_3d(&tmV, 64 * hf, ng, nx.k0);
          }
        }
      }
      if (!ok && even) {  // let this pair's copies in flight land before the CTAs exit
        mbar_wait_drain_cluster(b_kv, 0);
        for (int i = issued_qs > 2 ? issued_qs - 2 : 0; i < issued_qs; ++i)
          mbar_wait_drain_cluster(b_qsfull + 8 * (i & 1), (i >> 1) & 1);
        if (issued_dop > 0) mbar_wait_drain_cluster(b_dopfull, (issued_dop - 1) & 1);
        if (issued_dov > 0) mbar_wait_drain_cluster(b_dovfull, (issued_dov - 1) & 1);
        if (issued_qk > 0) mbar_wait_drain_cluster(b_qkfull, (issued_qk - 1) & 1);
      }
    } else if (warp == 1 && lane == 0 && even && npairs > 0) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      // Operand descriptors are the base's plus compile-time constants (one add
      // each): K-major operands lbo 16, MN-major lbo 16384 (a single 64-column
      // block per CTA).  The odd CTA's operands sit at the same offsets.
      const uint64_t d0 = sdesc_sw128(s0, 0, 1024);
      auto issue_s = [&](int i) {  // S^T_i = K Q_i^T
        const uint64_t db = opaque(d0);
        const uint64_t dq = sdesc_at(db, (uint32_t)(i & 1) * 16384, 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_pair(tmem + C::tS, sdesc_at(db, C::kK + (kk >> 2) * 16384 + (kk & 3) * 32, 16),
                       sdesc_at(dq, C::kQS + (kk >> 2) * 8192 + (kk & 3) * 32, 16), C::kIdescS, kk > 0);
        umma_commit_pair_both(b_s);
      };
      auto issue_dp = [&]() {  // dP^T = V dO^T
        const uint64_t db = opaque(d0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_pair(tmem + C::tP, sdesc_at(db, C::kV + (kk >> 2) * 16384 + (kk & 3) * 32, 16),
                       sdesc_at(db, C::kDOP + (kk >> 2) * 8192 + (kk & 3) * 32, 16), C::kIdescS, kk > 0);
        umma_commit_pair_both(b_dp);
        umma_commit_pair_both(b_dopempty);
      };
      bool ok = mbar_wait_cluster(b_kv, 0, ab, 235);
      if (ok) {
        ok = mbar_wait_cluster(b_qsfull, 0, ab, 236) && mbar_wait_cluster(b_dopfull, 0, ab, 237);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp();
        }
      }
      for (int i = 0; i < npairs && ok; ++i) {
        const int st = i & 1;
        const uint32_t pi = i & 1;
        const uint64_t db = opaque(d0);
        // dV += P^T dO once P_i is packed in both CTAs (A from tensor memory:
        // query columns 0-63 in columns [0,32) of the S region, 64-127 in [64,96))
        if (!mbar_wait_cluster(b_p, pi, ab, 238)) { ok = false; break; }
        if (i > 0 && i % C::kChain == 0) {  // the previous dV/dK chain has been flushed
          if (!mbar_wait_cluster(b_kvf, ((i / C::kChain) - 1) & 1, ab, 239)) { ok = false; break; }
        }
        if (!mbar_wait_cluster(b_dovfull, pi, ab, 240)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_pair(tmem + C::tdV, tmem + C::tS + (kk >> 2) * 64 + (kk & 3) * 8,
                       sdesc_at(db, C::kDOV + kk * 2048, 16384), C::kIdescG, (i % C::kChain > 0 || kk > 0) ? 1u : 0u);
        umma_commit_pair_both(b_dovempty);
        // S_{i+1} right behind dV_i, the last reader of P_i in the S region
        if (i + 1 < npairs) {
          if (!mbar_wait_cluster(b_qsfull + 8 * (st ^ 1), ((i + 1) >> 1) & 1, ab, 241)) { ok = false; break; }
          tc_fence_after();
          issue_s(i + 1);
        }
        // dQ_i = dS K over both key tiles, then dK += dS^T Q, once dS_i is in
        // both CTAs' shared and tensor memory
        if (!mbar_wait_cluster(b_pr, pi, ab, 242)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          umma_ss_pair(tmem + C::tQ, sdesc_at(db, C::kR + (kk >> 3) * 16384 + (kk & 7) * 2048, 16384),
                       sdesc_at(db, C::kKB + (kk >> 3) * 16384 + (kk & 7) * 2048, 16384), C::kIdescQ, kk > 0);
        umma_commit_pair_both(b_dq);
        if (!mbar_wait_cluster(b_qkfull, pi, ab, 243)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_pair(tmem + C::tdK, tmem + C::tP + (kk >> 2) * 96 + (kk & 3) * 8,
                       sdesc_at(db, C::kQK + kk * 2048, 16384), C::kIdescG, (i % C::kChain > 0 || kk > 0) ? 1u : 0u);
        umma_commit_pair_both(b_qkempty);
        umma_commit_pair_both(b_qsempty + 8 * st);
        umma_commit_pair_both(b_dsf);
        // dP_{i+1} once dQ_i has left the region and dO_{i+1} has landed
        if (i + 1 < npairs) {
          if (!mbar_wait_cluster(b_dqf, pi, ab, 244)) { ok = false; break; }
          if (!mbar_wait_cluster(b_dopfull, pi ^ 1, ab, 245)) { ok = false; break; }
          tc_fence_after();
          issue_dp();
        }
      }
      if (!ok) {  // let issued MMAs finish before tensor memory is released
        umma_commit_pair_own(b_drain);
        mbar_wait_drain_cluster(b_drain, 0);
      }
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;");
    // ------------------------------------------------------------ compute warpgroups
    // Warpgroup w takes query columns [64w, 64w + 64) of S^T/dP^T (TMEM lanes =
    // this CTA's keys) and head columns [64w, 64w + 64) of the final dK and dV.
    const int wg = (warp - 4) >> 2;
    const int tid = threadIdx.x - 128 * (1 + wg);
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t tS = tmem_addr(tmem, lane_base, C::tS);
    const uint32_t tP = tmem_addr(tmem, lane_base, C::tP);
    const int k0 = it.k0, k1 = it.k1;
    const int krow = k0 + tid;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2), scale2 = f2_pack(p.scale, p.scale);
    // dS^T rows of this warpgroup's query columns go to CTA wg's buffer for key
    // tile `rank` (its A operand of dQ for these keys), with cluster stores
    const uint32_t row_addr = mapa_shared(s0 + C::kR + rank * 16384 + tid * 128, (uint32_t)wg);
    const bool valid = krow < k1;
    float* dv_row = p.dv_acc + ((size_t)krow * p.Hkv + g) * D + wg * 64;
    float* dk_row = p.dk_acc + ((size_t)krow * p.Hkv + g) * D + wg * 64;
    auto flush_dkdv = [&]() {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t t = tmem_addr(tmem, lane_base, (which == 0 ? C::tdV : C::tdK) + wg * 64);
        float* dst = which == 0 ? dv_row : dk_row;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
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
      need_mask = (k1 - k0 < 128) || (q0 + 128 > qe) || (q0 < qlo) || (p.causal && k1 - 1 > q0);
      cmin = (krow >= k1) ? 128 : max(qlo - q0, p.causal ? krow - q0 : 0);
      cmax = qe - q0;  // exclusive
    };
    uint64_t pf[32];  // scale P^T of the current pair (packed fp32 pairs, masked), for its dS phase
    auto p_phase = [&](int i) -> bool {
      if (!wait_warp(b_s, i & 1, 250)) return false;
      tc_fence_after();
      bool need_mask;
      int cmin, cmax;
      vis(i, need_mask, cmin, cmax);
      const float4* sl4 = reinterpret_cast<const float4*>(stat + (i & 1) * 256);
      uint32_t r[2][32];
      tmem_ld32(tS + 64 * wg, r[0]);
      tmem_ld32(tS + 64 * wg + 32, r[1]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      uint32_t w0[16], w1[16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = 64 * wg + 32 * c + 2 * x;
          const float4 l4 = sl4[c0 >> 2];  // -LSE log2e of 4 columns
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
      if (lane == 0) arrive_lead(b_p);
      return true;
    };
    // dS^T = scale P^T (dP^T - Delta): packed into this warpgroup's columns of
    // the dP region (dK's A) and stored to CTA wg's dS buffer (dQ's A), once
    // dQ_{i-1} and dK_{i-1} have read the previous one
    auto ds_phase = [&](int i) -> bool {
      if (!wait_warp(b_dp, i & 1, 251)) return false;
      tc_fence_after();
      const float4* sl4 = reinterpret_cast<const float4*>(stat + (i & 1) * 256);
      uint32_t r[2][32];
      tmem_ld32(tP + 64 * wg, r[0]);
      tmem_ld32(tP + 64 * wg + 32, r[1]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      uint32_t w[2][16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = 64 * wg + 32 * c + 2 * x;
          const float4 d4 = sl4[32 + (c0 >> 2)];  // -Delta of 4 columns
          const uint64_t nd = (x & 1) ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
          float d0, d1;
          f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(r[c][2 * x]), __uint_as_float(r[c][2 * x + 1])), nd),
                           pf[16 * c + x]),
                    d0, d1);
          w[c][x] = pack_bf16x2(d0, d1);
        }
      }
      // dP_i has been read (and dK_{i-1}, which read the packed dS_{i-1}, ran
      // before dP_i): the packed dS_i goes to columns [0,32) (warpgroup 0) or
      // [96,128) (warpgroup 1) of the region
      tmem_st16(tP + 96 * wg, w[0]);
      tmem_st16(tP + 96 * wg + 16, w[1]);
      tmem_st_wait();
      tc_fence_before();
      if (i > 0 && !wait_warp(b_dsf, (i - 1) & 1, 252)) return false;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const int piece = c * 4 + pc;
          st_cluster_v4(row_addr + ((piece ^ (tid & 7)) << 4), w[c][4 * pc], w[c][4 * pc + 1], w[c][4 * pc + 2],
                        w[c][4 * pc + 3]);
        }
      fence_proxy_async_cluster();  // the pair's tensor core reads these
      __syncwarp();
      if (lane == 0) arrive_lead(b_pr);
      return true;
    };
    bool ok = npairs == 0 || p_phase(0);
    for (int i = 0; i < npairs && ok; ++i) {
      ok = ds_phase(i);
      if (ok && i + 1 < npairs) ok = p_phase(i + 1);
    }
    // every MMA of the pair is done once dQ and dK of the last pair are
    if (ok && npairs > 0 && wait_warp(b_dsf, (npairs - 1) & 1, 253)) {
      tc_fence_after();
      flush_dkdv();
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
    // ------------------------------------------------------------ dQ warpgroup
    // This CTA's dQ rows: lanes [0,64) hold its 64 query rows for head columns
    // [0,64), lanes [64,128) the same rows for columns [64,128), 64 tensor-memory
    // columns each.  Warp w: rows 32 (w & 1) .. + 32, head columns 64 (w >> 1)
    // .. + 64, staged 32 columns at a time (4 KB) and added with bulk tensor
    // reductions.  Rows outside the query range carry exact zeros.
    const int tid = threadIdx.x - 384;
    const int wq = warp & 3;
    const uint32_t lane_base = (uint32_t)wq * 32;
    const uint32_t tQ = tmem_addr(tmem, lane_base, C::tQ);
    const uint32_t wbuf = s0 + C::kStg + (uint32_t)wq * 4096;
    const uint32_t row = (uint32_t)lane * 128;
    const bool lead_lane = lane == 0;
    const int col0 = 64 * (wq >> 1), row0 = 64 * (int)rank + 32 * (wq & 1);
    for (int j = 0; j < npairs; ++j) {
      if (!wait_warp(b_dq, j & 1, 260)) break;
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(tQ, r[0]);
      tmem_ld32(tQ + 32, r[1]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_lead(b_dqf);  // dQ_j has left tensor memory
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (lead_lane) bulk_wait_read();  // the buffer's previous box has been read
        __syncwarp();
#pragma unroll
        for (int pc = 0; pc < 8; ++pc)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(wbuf + row + ((pc ^ (lane & 7)) << 4)),
                       "r"(r[k][4 * pc]), "r"(r[k][4 * pc + 1]), "r"(r[k][4 * pc + 2]), "r"(r[k][4 * pc + 3])
                       : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lead_lane) {
          tma_reduce_add_3d(&tmDQ, wbuf, col0 + 32 * k, pl.head(j), pl.start(j) + row0);
          bulk_commit();
        }
      }
      // pair j closed a dV/dK chain and more pairs follow: add the chain into
      // the fp32 accumulators (here lanes = this CTA's keys)
      if ((j + 1) % C::kChain == 0 && j + 1 < npairs) {
        if (!wait_warp(b_dsf, j & 1, 261)) break;  // dK_j is done too
        tc_fence_after();
        const int krow = it.k0 + tid;
        const bool valid = krow < it.k1;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t t = tmem_addr(tmem, lane_base, which == 0 ? C::tdV : C::tdK);
          float* dst = (which == 0 ? p.dv_acc : p.dk_acc) + ((size_t)krow * p.Hkv + g) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(t + 32 * c, rr);
            tmem_ld_wait();
            reg_fence32(rr);
            if (valid) {
#pragma unroll
              for (int x = 0; x < 8; ++x)
                red_add_v4(dst + 32 * c + 4 * x, __uint_as_float(rr[4 * x]), __uint_as_float(rr[4 * x + 1]),
                           __uint_as_float(rr[4 * x + 2]), __uint_as_float(rr[4 * x + 3]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_lead(b_kvf);
      }
    }
    if (lead_lane) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while the pair's MMAs or cluster stores may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd_step_pair(const CUtensorMap& tq, const CUtensorMap& tq64, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdo64,
                                 const CUtensorMap& tl, const CUtensorMap& td, const CUtensorMap& tdq,
                                 const BwdParams& p, int num_items, cudaStream_t stream) {
  auto kern = ring_bwd_pair_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::kSmem);
  if (e != cudaSuccess) return e;
  if (num_items <= 0) return cudaSuccess;
  if (num_items & 1) return cudaErrorInvalidValue;  // items come in pairs of key tiles
  BwdParams q = p;  // one CTA per SM: the stride to the CTA that follows on an SM
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  q.next_cta = sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_items, 1, 1);
  cfg.blockDim = dim3(512, 1, 1);
  cfg.dynamicSmemBytes = PairCfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tq, tq64, tk, tv, tdo, tdo64, tl, td, tdq, q);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ra
