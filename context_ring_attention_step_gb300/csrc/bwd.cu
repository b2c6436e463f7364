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
// Warp roles (384 threads):
//   warp 0      producer: K, V once; then Q_i, dO_i (TMA) and the LSE/Delta
//               slices of each pair into a two-stage ring
//   warp 1      TMEM owner + single-thread UMMA issuer
//   warps 4-11  two compute warpgroups, each on half of the 128 query columns
//               (P^T, dS^T) and half of the head dimension (dQ read-out and
//               bulk reduction, final dK/dV flush)
// Tensor memory: dV [0,D), dK [D,2D), S^T/P^T [2D,2D+128), dP^T/dS^T/dQ after.
// P^T and dS^T (bf16, two per column) overwrite columns [0,32) and [64,96) of
// S^T and dP^T (each warpgroup packs into its own columns) and feed the dV and
// dK MMAs from tensor memory; dS^T is also written to shared memory
// (MN-major, 128-byte swizzle) as the A operand of the dQ MMA.
#include "ring_attn_internal.h"
#include "tc.cuh"

namespace ra {
namespace {

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kStage0 = 2 * kTile;          // two stages of {Q, dO}
  static constexpr int kDS = kStage0 + 4 * kTile;    // dS^T, 128 x 128 bf16
  static constexpr int kStat = kDS + 32768;          // per stage: lse2[128], delta[128] (TMA)
  static constexpr int kBar = kStat + 2 * 1024;
  static constexpr int kSmem = kBar + 256;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, false, true);   // dV, dK: A tmem, B MN-major
  static constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, true, true);    // dQ: A, B MN-major
  static constexpr uint32_t tdV = 0, tdK = D, tS = 2 * D, tP = 2 * D + 128;
};

// Query tiles of the CTA's pairs.  Tiles of a range start at the range start
// rounded down to a multiple of 4, so the LSE/Delta slice of every tile is a
// 16-byte aligned TMA load; columns before the range start are masked.
struct PairList {
  int qb0, qe0, qb1, qe1, n0, nt, G, hbase;
  __device__ __forceinline__ int tile(int i) const { return i % nt; }
  __device__ __forceinline__ int head(int i) const { return hbase + i / nt; }
  __device__ __forceinline__ int start(int i) const {
    const int t = tile(i);
    return t < n0 ? (qb0 & ~3) + 128 * t : (qb1 & ~3) + 128 * (t - n0);
  }
  __device__ __forceinline__ int lo(int i) const { return tile(i) < n0 ? qb0 : qb1; }
  __device__ __forceinline__ int end(int i) const { return tile(i) < n0 ? qe0 : qe1; }
};

__device__ __forceinline__ int ceil128(int a, int b) { return b > a ? (b - a + 127) / 128 : 0; }

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D>
__global__ void __launch_bounds__(384, 1)
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
  const uint32_t sK = s0 + C::kK, sV = s0 + C::kV, sSt = s0 + C::kStage0, sDS = s0 + C::kDS;
  float* stat = reinterpret_cast<float*>(smem + C::kStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  const uint32_t b_kv = smem_u32(bars + 0);
  const uint32_t b_full = smem_u32(bars + 1);    // [2]
  const uint32_t b_empty = smem_u32(bars + 3);   // [2]
  const uint32_t b_s = smem_u32(bars + 5);
  const uint32_t b_dp = smem_u32(bars + 6);
  const uint32_t b_pr = smem_u32(bars + 7);      // P^T, dS^T written (128 arrivals)
  const uint32_t b_dq = smem_u32(bars + 8);      // dQ_i in TMEM (and all earlier MMAs done)
  const uint32_t b_dqf = smem_u32(bars + 9);     // dQ_i read out (128 arrivals)
  const uint32_t b_drain = smem_u32(bars + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
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
    mbar_init(b_full, 1); mbar_init(b_full + 8, 1);
    mbar_init(b_empty, 1); mbar_init(b_empty + 8, 1);
    mbar_init(b_s, 1); mbar_init(b_dp, 1);
    mbar_init(b_pr, 256);
    mbar_init(b_dq, 1);
    mbar_init(b_dqf, 256);
    mbar_init(b_drain, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmL); tma_prefetch_desc(&tmD);
      mbar_expect_tx(b_kv, 2 * C::kTile);
      for (int hf = 0; hf < D / 64; ++hf) {
        tma_load_3d(sK + hf * 16384, &tmK, b_kv, 64 * hf, g, it.k0);
        tma_load_3d(sV + hf * 16384, &tmV, b_kv, 64 * hf, g, it.k0);
      }
      for (int i = 0; i < npairs; ++i) {
        const int st = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(b_empty + 8 * st, ph ^ 1, ab, 201)) { ok = false; break; }
        const int h = pl.head(i), q0 = pl.start(i);
        const uint32_t sq = sSt + st * 2 * C::kTile, sdo = sq + C::kTile;
        const uint32_t sl = smem_u32(stat + st * 256);
        mbar_expect_tx(b_full + 8 * st, 2 * C::kTile + 2 * 512);
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_3d(sq + hf * 16384, &tmQ, b_full + 8 * st, 64 * hf, h, q0);
          tma_load_3d(sdo + hf * 16384, &tmDO, b_full + 8 * st, 64 * hf, h, q0);
        }
        // LSE (log2 units) and Delta of the tile's 128 query columns
        tma_load_2d(sl, &tmL, b_full + 8 * st, q0, h);
        tma_load_2d(sl + 512, &tmD, b_full + 8 * st, q0, h);
        ++issued;
      }
      if (!ok) {
        mbar_wait_drain(b_kv, 0);
        for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
          mbar_wait_drain(b_full + 8 * (i & 1), (i >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per pair i:  [dQ_{i-1} read out] dP_i | [P_i, dS_i written] dV_i, S_{i+1}, dK_i, dQ_i.
    // S_{i+1} goes right after dV_i (the last reader of P_i in the S region), so
    // the next pair's P phase overlaps dK_i and dQ_i.
    if (lane == 0) {
      auto issue_s = [&](int i) {  // S^T_i = K Q_i^T
        const uint32_t sq = sSt + (i & 1) * 2 * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tmem + C::tS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sq + off, 16, 1024), C::kIdescS,
                  kk > 0);
        }
        umma_commit(b_s);
      };
      bool ok = mbar_wait(b_kv, 0, ab, 202);
      if (ok && npairs > 0) {
        ok = mbar_wait(b_full, 0, ab, 203);
        if (ok) {
          tc_fence_after();
          issue_s(0);
        }
      }
      for (int i = 0; i < npairs && ok; ++i) {
        const int st = i & 1;
        const uint32_t pi = i & 1;
        const uint32_t sq = sSt + st * 2 * C::kTile, sdo = sq + C::kTile;
        // dP^T = V dO^T, once dQ_{i-1} has left this tensor-memory region
        if (i > 0) {
          if (!mbar_wait(b_dqf, pi ^ 1, ab, 204)) { ok = false; break; }
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tmem + C::tP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sdo + off, 16, 1024), C::kIdescS,
                  kk > 0);
        }
        umma_commit(b_dp);
        if (!mbar_wait(b_pr, pi, ab, 205)) { ok = false; break; }
        tc_fence_after();
        // dV += P^T dO   (A from tensor memory: packed query columns 0-63 in
        // columns [0,32) of the S region, 64-127 in columns [64,96); B MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + C::tdV, tmem + C::tS + (kk >> 2) * 64 + (kk & 3) * 8,
                  sdesc_sw128(sdo + kk * 2048, 16384, 1024), C::kIdescG, (i > 0 || kk > 0) ? 1u : 0u);
        if (i + 1 < npairs) {
          if (!mbar_wait(b_full + 8 * (st ^ 1), ((i + 1) >> 1) & 1, ab, 203)) { ok = false; break; }
          tc_fence_after();
          issue_s(i + 1);
        }
        // dK += dS^T Q
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + C::tdK, tmem + C::tP + (kk >> 2) * 64 + (kk & 3) * 8,
                  sdesc_sw128(sq + kk * 2048, 16384, 1024), C::kIdescG, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(b_empty + 8 * st);
        // dQ_i = dS K   (A = dS from shared memory, MN-major; B = K, MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + C::tP, sdesc_sw128(sDS + kk * 2048, 16384, 1024), sdesc_sw128(sK + kk * 2048, 16384, 1024),
                  C::kIdescQ, kk > 0);
        umma_commit(b_dq);
      }
      if (!ok) {
        umma_commit(b_drain);
        mbar_wait_drain(b_drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute warpgroups
    // Two warpgroups split every 128-column tile: warpgroup w takes query
    // columns [64w, 64w + 64) of S^T/dP^T, and head-dim columns [D/2 w, D/2 (w+1))
    // of dQ, dK and dV.  TMEM lanes: key rows for S^T/dP^T/dK/dV, query rows for dQ.
    const int wg = (warp - 4) >> 2;
    const int tid = threadIdx.x - 128 * (1 + wg);
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t tS = tmem_addr(tmem, lane_base, C::tS);
    const uint32_t tP = tmem_addr(tmem, lane_base, C::tP);
    const int krow = it.k0 + tid;
    const float sl2 = p.scale_log2, scale = p.scale;
    constexpr int DH = D / 2;  // head-dim columns per warpgroup
    bool ok = true;
    // dQ_j, this warpgroup's head-dim half: read out of tensor memory, staged
    // 16 columns at a time and added into the fp32 accumulator by bulk tensor
    // reductions.  Each warp stages only its own 32 rows, in the 4 KB of the
    // dS buffer that it also writes dS^T to, split into two 2 KB halves used
    // alternately (64-byte swizzle): a round waits only for the reads of the
    // round before last, and no warp waits for another.  Rows outside the
    // query range carry exact zeros (their dS columns are masked); rows past T
    // are clipped by the tensor map.
    const uint32_t row_addr = sDS + wg * 16384 + tid * 128;
    const uint32_t warp_box = sDS + wg * 16384 + (tid & ~31) * 128;
    const uint32_t half_row = (uint32_t)lane * 64;
    const uint32_t swz64 = (uint32_t)((lane >> 1) & 3);
    const bool lead = lane == 0;
    // all lanes of a warp take the same branch after a bounded wait
    auto wait_warp = [&](uint32_t bar, uint32_t parity, int site) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, site)) != 0;
    };
    auto dq_out = [&](int j) -> bool {
      if (!wait_warp(b_dq, j & 1, 220)) return false;
      tc_fence_after();
      uint32_t r[DH / 32][32];
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) tmem_ld32(tP + wg * DH + 32 * c, r[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) reg_fence32(r[c]);
      tc_fence_before();
      mbar_arrive(b_dqf);
#pragma unroll
      for (int c = 0; c < DH / 16; ++c) {
        const uint32_t buf = warp_box + (c & 1) * 2048;
        if (lead) bulk_wait_read_all_but_one();  // this half's previous box has been read
        __syncwarp();
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const int x = 16 * (c & 1) + 4 * pc;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + half_row + ((pc ^ swz64) << 4)),
                       "r"(r[c >> 1][x]), "r"(r[c >> 1][x + 1]), "r"(r[c >> 1][x + 2]), "r"(r[c >> 1][x + 3])
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lead) {
          tma_reduce_add_3d(&tmDQ, buf, wg * DH + 16 * c, pl.head(j), pl.start(j) + (tid & ~31));
          bulk_commit();
        }
      }
      return true;
    };
    for (int i = 0; i < npairs && ok; ++i) {
      const int st = i & 1;
      const uint32_t pi = i & 1;
      const int q0 = pl.start(i), qlo = pl.lo(i), qe = pl.end(i);
      const float4* sl4 = reinterpret_cast<const float4*>(stat + st * 256);
      const bool need_mask =
          (it.k1 - it.k0 < 128) || (q0 + 128 > qe) || (q0 < qlo) || (p.causal && it.k1 - 1 > q0);
      // visible query columns c satisfy  qlo <= q0 + c < qe  and (causal) krow <= q0 + c
      const int cmin = (krow >= it.k1) ? 128 : max(qlo - q0, p.causal ? krow - q0 : 0);
      const int cmax = qe - q0;  // exclusive
      // ---- P^T = exp2(S^T scale log2e - LSE log2e) on columns [64 wg, 64 wg + 64)
      if (!wait_warp(b_s, pi, 210)) { ok = false; break; }
      tc_fence_after();
      uint32_t pk[32];
      {
        uint32_t r[2][32];
        tmem_ld32(tS + 64 * wg, r[0]);
        tmem_ld32(tS + 64 * wg + 32, r[1]);
        tmem_ld_wait();
        reg_fence32(r[0]);
        reg_fence32(r[1]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int c0 = 64 * wg + 32 * c + 2 * x;
            const float4 l4 = sl4[c0 >> 2];  // broadcast read of 4 columns' LSE
            const float la = (x & 1) ? l4.z : l4.x, lb = (x & 1) ? l4.w : l4.y;
            float p0 = ex2_approx(fmaf(__uint_as_float(r[c][2 * x]), sl2, -la));
            float p1 = ex2_approx(fmaf(__uint_as_float(r[c][2 * x + 1]), sl2, -lb));
            if (need_mask) {
              if (c0 < cmin || c0 >= cmax) p0 = 0.f;
              if (c0 + 1 < cmin || c0 + 1 >= cmax) p1 = 0.f;
            }
            pk[16 * c + x] = pack_bf16x2(p0, p1);
          }
        }
        // packed P^T goes to the first half of this warpgroup's own 64 columns
        // (never into the other warpgroup's columns, which it may not have read yet)
        uint32_t w0[16], w1[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) { w0[x] = pk[x]; w1[x] = pk[16 + x]; }
        tmem_st16(tS + 64 * wg, w0);
        tmem_st16(tS + 64 * wg + 16, w1);
      }
      // ---- dQ of the previous pair (frees the dP region for dP^T_i)
      if (i > 0 && !dq_out(i - 1)) { ok = false; break; }
      // ---- dS^T = scale P^T (dP^T - Delta)
      if (!wait_warp(b_dp, pi, 211)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t r[2][32];
        tmem_ld32(tP + 64 * wg, r[0]);
        tmem_ld32(tP + 64 * wg + 32, r[1]);
        tmem_ld_wait();
        reg_fence32(r[0]);
        reg_fence32(r[1]);
        // this warpgroup's 64 query columns are chunk `wg` of the MN-major dS tile
        uint32_t w[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int c0 = 64 * wg + 32 * c + 2 * x;
            const uint32_t pp = pk[16 * c + x];
            const float4 d4 = sl4[32 + (c0 >> 2)];  // broadcast read of 4 columns' Delta
            const float da = (x & 1) ? d4.z : d4.x, db = (x & 1) ? d4.w : d4.y;
            const float d0 = bf16lo(pp) * (__uint_as_float(r[c][2 * x]) - da) * scale;
            const float d1 = bf16hi(pp) * (__uint_as_float(r[c][2 * x + 1]) - db) * scale;
            w[c][x] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tP + 64 * wg + 16 * c, w[c]);
        }
        // the TMA must have read this warp's staged dQ rows before they are rewritten
        if (lead) bulk_wait_read();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            const int piece = c * 4 + pc;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row_addr + ((piece ^ (tid & 7)) << 4)),
                         "r"(w[c][4 * pc]), "r"(w[c][4 * pc + 1]), "r"(w[c][4 * pc + 2]), "r"(w[c][4 * pc + 3])
                         : "memory");
          }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(b_pr);
    }
    if (ok && npairs > 0) ok = dq_out(npairs - 1);  // also: every MMA of the CTA is done
    if (lead) bulk_wait_all();
    if (ok && npairs > 0) {
      const bool valid = krow < it.k1;
      float* dv_row = p.dv_acc + ((size_t)krow * p.Hkv + g) * D + wg * DH;
      float* dk_row = p.dk_acc + ((size_t)krow * p.Hkv + g) * D + wg * DH;
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
    }
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
  kern<<<(unsigned)grid, 384, BwdCfg<D>::kSmem, stream>>>(tq, tk, tv, tdo, tl, td, tdq, p);
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
