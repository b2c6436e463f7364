// bwd256.cu -- one ring step of the backward pass for head_dim 256 on tcgen05
// tensor cores.
//
// S and dP reduce over all 256 columns, so a CTA keeps its whole K and V tile
// (128 keys x 256 columns, 64 KB each) in shared memory.  The gradients split
// by columns: dV = P^T dO, dK = dS^T Q and dQ = dS K each take one 128-column
// half of dO, Q or K.  So two CTAs share a 128-key tile of one key/value head,
// CTA c owning columns [128c, 128c + 128) of dK, dV (accumulated in tensor
// memory over the CTA's pairs) and of the dQ contributions.  Both recompute
// S^T = K Q^T and dP^T = V dO^T.  Query tiles are 64 rows, single-buffered:
// with K and V resident that is what shared memory holds.  dQ is formed
// transposed, dQ^T = K_c^T dS^T (tensor-memory lanes = the 128 columns of the
// half, 64 query columns), so every MMA has M = 128.
//
// Per pair (query head, 64-row query tile), with LSE and Delta of its rows:
//   S^T = K Q^T, P^T = exp(scale S^T - LSE), dP^T = V dO^T,
//   dS^T = scale P^T (dP^T - Delta),
//   dV_c += P^T dO_c,  dK_c += dS^T Q_c,  dQ_c^T = K_c^T dS^T
// (P^T from the unrounded fp32 P for dS; the bf16-rounded P feeds the dV MMA
// from tensor memory).
//
// Warp roles (512 threads):
//   warp 0       producer: K, V once; per pair Q_i with its LSE/Delta slices and dO_i,
//                each in two column halves released separately
//   warp 1       TMEM owner + single-thread UMMA issuer
//   warps 4-11   two compute warpgroups, each on half of the 64 query columns:
//                P^T (tensor memory), dS^T (shared memory); TMEM lanes = keys;
//                every kChain pairs, and at the end, they add dK_c, dV_c into the
//                fp32 accumulators (each warpgroup half of the columns)
//   warps 12-15  dQ: read dQ_c^T out of tensor memory (lanes = columns), stage it
//                per warp as 32 query rows x 32 columns and add it into the fp32
//                accumulator with bulk tensor reductions
// Tensor memory: dV_c [0,128), dK_c [128,256), S^T/P^T [256,320), dP^T [320,384),
// dQ_c^T [384,448).  P^T (bf16, two per column) overwrites columns [0,16) and
// [32,48) of S^T, each warpgroup in its own columns.
#include "ring_attn_internal.h"
#include "tc.cuh"

namespace ra {
namespace {

namespace b256 {
constexpr int kD = 256;
constexpr int kK = 0;              // K tile: 4 boxes of 64 columns x 128 keys (16 KB each)
constexpr int kV = 65536;          // V tile: same
constexpr int kQ = 131072;         // Q tile: 4 boxes of 64 columns x 64 rows (8 KB each)
constexpr int kDO = 163840;        // dO tile: same
constexpr int kDS = 196608;        // dS^T: 128 keys x 64 queries bf16, 128-byte swizzle
constexpr int kStg = 212992;       // dQ staging: 4 warps x (32 rows x 32 fp32)
constexpr int kStat = 229376;      // lse2[64], delta[64]
constexpr int kBar = kStat + 512;
constexpr int kSmem = kBar + 256;  // 230144 bytes
constexpr uint32_t tdV = 0, tdK = 128, tS = 256, tP = 320, tQ = 384;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);   // S^T, dP^T
constexpr uint32_t kIdescG = idesc_bf16_f32(128, 128, false, true);   // dV, dK: B MN-major
constexpr uint32_t kIdescQ = idesc_bf16_f32(128, 64, true, true);     // dQ^T: A, B MN-major
constexpr int kChain = 256;  // pairs per dV/dK chain in tensor memory (bounds the fp32 drift)
}  // namespace b256

struct Pairs64 {
  int qb0, qe0, qb1, qe1, n0, nt, hbase;
  __device__ __forceinline__ int tile(int i) const { return i % nt; }
  __device__ __forceinline__ int head(int i) const { return hbase + i / nt; }
  __device__ __forceinline__ int start(int i) const {
    const int t = tile(i);
    return t < n0 ? (qb0 & ~3) + 64 * t : (qb1 & ~3) + 64 * (t - n0);
  }
  __device__ __forceinline__ int lo(int i) const { return tile(i) < n0 ? qb0 : qb1; }
  __device__ __forceinline__ int end(int i) const { return tile(i) < n0 ? qe0 : qe1; }
};

__device__ __forceinline__ int ceil64(int a, int b) { return b > a ? (b - a + 63) / 64 : 0; }

__device__ __forceinline__ void red_add4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__global__ void __launch_bounds__(512, 1)
    ring_bwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                         const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using namespace b256;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (*reinterpret_cast<volatile int*>(p.status) != 0) return;
  if ((smem_u32(smem) & 1023u) != 0) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0) atomicCAS(p.status, 0, 298);
    return;
  }
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + kK, sV = s0 + kV, sQ = s0 + kQ, sDO = s0 + kDO, sDS = s0 + kDS, sStg = s0 + kStg;
  float* stat = reinterpret_cast<float*>(smem + kStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBar);
  // Q and dO tiles go in two column halves with barriers of their own: the
  // half a CTA does not use for dV/dK ("other") is free as soon as S (or dP)
  // has read it, so the next tile's half loads early and S_{i+1} starts on it
  // while the own half (freed by dK / dV) is still coming.
  const uint32_t b_kv = smem_u32(bars + 0);
  const uint32_t b_qfull = smem_u32(bars + 1);    // [2] Q_i column half landed (own half: + LSE/Delta)
  const uint32_t b_qempty = smem_u32(bars + 3);   // [2] Q column half released (other: after S_i; own: after dK_i)
  const uint32_t b_dofull = smem_u32(bars + 5);   // [2] dO_i column half landed
  const uint32_t b_doempty = smem_u32(bars + 7);  // [2] dO column half released (other: after dP_i; own: after dV_i)
  const uint32_t b_s = smem_u32(bars + 9);        // S^T_i in tensor memory
  const uint32_t b_dp = smem_u32(bars + 10);      // dP^T_i in tensor memory
  const uint32_t b_p = smem_u32(bars + 11);       // P^T_i packed in tensor memory
  const uint32_t b_ds = smem_u32(bars + 12);      // dS^T_i written to shared memory
  const uint32_t b_dq = smem_u32(bars + 13);      // dQ_i^T in tensor memory
  const uint32_t b_dqf = smem_u32(bars + 14);     // dQ_i^T read out
  const uint32_t b_dsf = smem_u32(bars + 15);     // dK_i and dQ_i^T done (dS buffer free)
  const uint32_t b_drain = smem_u32(bars + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdItem it = p.items[blockIdx.x >> 1];
  const int half = blockIdx.x & 1;  // the 128 columns this CTA owns
  const int g = it.flags >> kHeadShift;
  Pairs64 pl;
  pl.qb0 = it.qb0; pl.qe0 = it.qe0; pl.qb1 = it.qb1; pl.qe1 = it.qe1;
  pl.n0 = ceil64(it.qb0 & ~3, it.qe0);
  pl.nt = pl.n0 + ceil64(it.qb1 & ~3, it.qe1);
  const int G = p.Hq / p.Hkv;
  pl.hbase = g * G;
  const int npairs = pl.nt * G;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(b_qfull + 8 * x, 1); mbar_init(b_qempty + 8 * x, 1);
      mbar_init(b_dofull + 8 * x, 1); mbar_init(b_doempty + 8 * x, 1);
    }
    mbar_init(b_s, 1); mbar_init(b_dp, 1);
    mbar_init(b_p, 8); mbar_init(b_ds, 8);  // one arrival per compute warp (two warpgroups)
    mbar_init(b_dq, 1); mbar_init(b_dqf, 4);
    mbar_init(b_dsf, 1);
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
  auto wait_warp = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, site)) != 0;
  };

  // Register split: 512 threads x 128 at launch.  Producer/MMA warpgroup 88
  // (its unrolled MMA loop spills below that), compute warpgroups 152, dQ
  // warpgroup 104: 128 x (88 + 2 x 152 + 104) = 63488 <= 65536.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      bool ok = true;
      int issued = 0;  // pairs whose four loads were all issued
      int partial = 0;  // loads issued for the pair in progress (0..4)
      const int own = half, oth = 1 - half;
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmL); tma_prefetch_desc(&tmD);
      mbar_expect_tx(b_kv, 2 * 65536);
      for (int b = 0; b < 4; ++b) {
        tma_load_3d(sK + b * 16384, &tmK, b_kv, 64 * b, g, it.k0);
        tma_load_3d(sV + b * 16384, &tmV, b_kv, 64 * b, g, it.k0);
      }
      // one column half (two 64-column boxes) of a 64-row Q or dO tile
      auto load_half = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int h, int q0) {
        for (int b = 0; b < 2; ++b) tma_load_3d(dst + (2 * x + b) * 8192, m, bar, 64 * (2 * x + b), h, q0);
      };
      for (int i = 0; i < npairs && ok; ++i) {
        const int h = pl.head(i), q0 = pl.start(i);
        const uint32_t ph = (uint32_t)(i & 1) ^ 1u;
        partial = 0;
        // in the order the previous pair releases them: Q other (after S),
        // dO other (after dP), dO own (after dV), Q own with LSE/Delta (after dK)
        if (!mbar_wait(b_qempty + 8 * oth, ph, ab, 241)) { ok = false; break; }
        mbar_expect_tx(b_qfull + 8 * oth, 16384);
        load_half(sQ, &tmQ, b_qfull + 8 * oth, oth, h, q0);
        ++partial;
        if (!mbar_wait(b_doempty + 8 * oth, ph, ab, 242)) { ok = false; break; }
        mbar_expect_tx(b_dofull + 8 * oth, 16384);
        load_half(sDO, &tmDO, b_dofull + 8 * oth, oth, h, q0);
        ++partial;
        if (!mbar_wait(b_doempty + 8 * own, ph, ab, 242)) { ok = false; break; }
        mbar_expect_tx(b_dofull + 8 * own, 16384);
        load_half(sDO, &tmDO, b_dofull + 8 * own, own, h, q0);
        ++partial;
        if (!mbar_wait(b_qempty + 8 * own, ph, ab, 241)) { ok = false; break; }
        mbar_expect_tx(b_qfull + 8 * own, 16384 + 2 * 256);
        load_half(sQ, &tmQ, b_qfull + 8 * own, own, h, q0);
        tma_load_2d(smem_u32(stat), &tmL, b_qfull + 8 * own, q0, h);
        tma_load_2d(smem_u32(stat + 64), &tmD, b_qfull + 8 * own, q0, h);
        partial = 0;
        ++issued;
      }
      {
        // the CTA that takes this SM next: its K/V tile into L2 now
        const long long nb = (long long)blockIdx.x + p.next_cta;
        if (ok && p.next_cta > 0 && nb < (long long)gridDim.x) {
          const BwdItem nx = p.items[nb >> 1];
          const int ng = nx.flags >> kHeadShift;
          for (int b = 0; b < 4; ++b) {
            tma_prefetch_l2_3d(&tmK, 64 * b, ng, nx.k0);
            tma_prefetch_l2_3d(&tmV, 64 * b, ng, nx.k0);
          }
        }
      }
      if (!ok) {  // drain this CTA's copies still in flight
        mbar_wait_drain(b_kv, 0);
        const uint32_t bars4[4] = {b_qfull + 8 * (uint32_t)oth, b_dofull + 8 * (uint32_t)oth,
                                   b_dofull + 8 * (uint32_t)own, b_qfull + 8 * (uint32_t)own};
        for (int x = 0; x < 4; ++x) {
          const int n = issued + (x < partial ? 1 : 0);  // loads issued on this barrier
          if (n > 0) mbar_wait_drain(bars4[x], (uint32_t)(n - 1) & 1u);
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      bool ok = npairs > 0 && mbar_wait(b_kv, 0, ab, 243);
      const uint32_t dO_c = sDO + (uint32_t)half * 16384, Q_c = sQ + (uint32_t)half * 16384;
      const uint32_t K_c = sK + (uint32_t)half * 32768;
      for (int i = 0; i < npairs && ok; ++i) {
        const uint32_t pi = (uint32_t)i & 1u;
        const bool chain_start = (i % kChain) == 0;
        // S^T = K Q^T and dP^T = V dO^T over the 256 columns, the other
        // column half first (it lands first), releasing it right away
        const int oth = 1 - half;
        auto s_half = [&](uint32_t d, uint32_t a, uint32_t bq, int x, bool first) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int gk = 8 * x + k;
            const uint32_t ko = (gk >> 2) * 16384 + (gk & 3) * 32, qo = (gk >> 2) * 8192 + (gk & 3) * 32;
            umma_ss(d, sdesc_sw128(a + ko, 16, 1024), sdesc_sw128(bq + qo, 16, 1024), kIdescS,
                    (first && k == 0) ? 0u : 1u);
          }
        };
        if (!mbar_wait(b_qfull + 8 * oth, pi, ab, 244)) { ok = false; break; }
        tc_fence_after();
        s_half(tmem + tS, sK, sQ, oth, true);
        umma_commit(b_qempty + 8 * oth);
        if (!mbar_wait(b_qfull + 8 * half, pi, ab, 244)) { ok = false; break; }
        tc_fence_after();
        s_half(tmem + tS, sK, sQ, half, false);
        umma_commit(b_s);
        if (!mbar_wait(b_dofull + 8 * oth, pi, ab, 245)) { ok = false; break; }
        tc_fence_after();
        s_half(tmem + tP, sV, sDO, oth, true);
        umma_commit(b_doempty + 8 * oth);
        if (!mbar_wait(b_dofull + 8 * half, pi, ab, 245)) { ok = false; break; }
        tc_fence_after();
        s_half(tmem + tP, sV, sDO, half, false);
        umma_commit(b_dp);
        // dV_c += P^T dO_c once P^T is packed (A from tensor memory: query
        // columns 0-31 in columns [0,16) of the S region, 32-63 in [32,48);
        // B MN-major, the half's two 64-column boxes 8 KB apart)
        if (!mbar_wait(b_p, pi, ab, 246)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts(tmem + tdV, tmem + tS + (kk >> 1) * 32 + (kk & 1) * 8, sdesc_sw128(dO_c + kk * 2048, 8192, 1024),
                  kIdescG, (!chain_start || kk > 0) ? 1u : 0u);
        umma_commit(b_doempty + 8 * half);
        // dK_c += dS^T Q_c once dS^T is in shared memory
        if (!mbar_wait(b_ds, pi, ab, 247)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tmem + tdK, sdesc_sw128(sDS + kk * 32, 16, 1024), sdesc_sw128(Q_c + kk * 2048, 8192, 1024),
                  kIdescG, (!chain_start || kk > 0) ? 1u : 0u);
        umma_commit(b_qempty + 8 * half);
        // dQ_c^T = K_c^T dS^T once the previous one has left tensor memory
        if (i > 0 && !mbar_wait(b_dqf, pi ^ 1u, ab, 248)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + tQ, sdesc_sw128(K_c + kk * 2048, 16384, 1024), sdesc_sw128(sDS + kk * 2048, 16384, 1024),
                  kIdescQ, kk > 0);
        umma_commit(b_dq);
        umma_commit(b_dsf);
      }
      if (!ok && npairs > 0) {  // let issued MMAs finish before tensor memory is released
        umma_commit(b_drain);
        mbar_wait_drain(b_drain, 0);
      }
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    // ------------------------------------------------------------ compute warpgroups
    // Two warpgroups split each tile's 64 query columns: warpgroup w takes
    // columns [32w, 32w + 32) of S^T/dP^T (TMEM lanes = key rows), packs P^T
    // into tensor-memory columns [32w, 32w + 16) of the S region and writes
    // 16-byte chunks [4w, 4w + 4) of each dS^T row; at the end each flushes
    // half of the 128 dK/dV columns.
    const int wg = (warp - 4) >> 2;
    const int tid = threadIdx.x - 128 * (1 + wg);
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t aS = tmem_addr(tmem, lane_base, tS + 32 * wg), aP = tmem_addr(tmem, lane_base, tP + 32 * wg);
    // packed P^T goes into this warpgroup's own S columns (never into the
    // other warpgroup's, which it may not have read yet)
    const uint32_t aPk = aS;
    const int krow = it.k0 + tid;
    const bool valid = krow < it.k1;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2), scale2 = f2_pack(p.scale, p.scale);
    const uint32_t row_addr = sDS + (uint32_t)tid * 128;
    auto flush_dkdv = [&]() {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t t = tmem_addr(tmem, lane_base, (which == 0 ? tdV : tdK) + 64 * wg);
        float* dst = (which == 0 ? p.dv_acc : p.dk_acc) + ((size_t)krow * p.Hkv + g) * kD + 128 * half + 64 * wg;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(t + 32 * c, r);
          tmem_ld_wait();
          reg_fence32(r);
          if (valid) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
              red_add4(dst + 32 * c + 4 * x, __uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                       __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
      }
    };
    uint64_t pf[16];  // P^T of this warpgroup's columns (packed fp32 pairs, masked), for its dS phase
    bool ok = true;
    for (int i = 0; i < npairs && ok; ++i) {
      const uint32_t pi = (uint32_t)i & 1u;
      // ---- P^T = exp2(S^T scale log2e - LSE log2e) on this warpgroup's 32 columns
      if (!wait_warp(b_s, pi, 250)) { ok = false; break; }
      tc_fence_after();
      const int q0 = pl.start(i), qlo = pl.lo(i), qe = pl.end(i);
      const int cmin = valid ? max(qlo - q0, p.causal ? krow - q0 : 0) : 64;
      const int cmax = qe - q0;  // exclusive
      {
        uint32_t r[32];
        tmem_ld32(aS, r);
        tmem_ld_wait();
        reg_fence32(r);
        const float4* l4 = reinterpret_cast<const float4*>(stat);  // -LSE log2e
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = 32 * wg + 2 * x;
          const float4 l = l4[c0 >> 2];
          const uint64_t nl = (x & 1) ? f2_pack(l.z, l.w) : f2_pack(l.x, l.y);
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])), sl2x2, nl), x0, x1);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (c0 < cmin || c0 >= cmax) p0 = 0.f;
          if (c0 + 1 < cmin || c0 + 1 >= cmax) p1 = 0.f;
          pf[x] = f2_pack(p0, p1);
          w[x] = pack_bf16x2(p0, p1);
        }
        tmem_st16(aPk, w);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p);
      // ---- dS^T = scale P^T (dP^T - Delta) to shared memory, once dK and dQ of
      // the previous pair have read the buffer
      if (!wait_warp(b_dp, pi, 251)) { ok = false; break; }
      tc_fence_after();
      uint32_t w[16];
      {
        uint32_t r[32];
        tmem_ld32(aP, r);
        tmem_ld_wait();
        reg_fence32(r);
        const float4* d4 = reinterpret_cast<const float4*>(stat + 64);  // -scale Delta
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = 32 * wg + 2 * x;
          const float4 d = d4[c0 >> 2];
          const uint64_t nd = (x & 1) ? f2_pack(d.z, d.w) : f2_pack(d.x, d.y);
          float v0, v1;
          f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])), scale2, nd), pf[x]), v0,
                    v1);
          w[x] = pack_bf16x2(v0, v1);
        }
      }
      tc_fence_before();  // dP^T is in registers
      if (i > 0 && !wait_warp(b_dsf, pi ^ 1u, 252)) { ok = false; break; }
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int chunk = 4 * wg + pc;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row_addr + ((chunk ^ (tid & 7)) << 4)),
                     "r"(w[4 * pc]), "r"(w[4 * pc + 1]), "r"(w[4 * pc + 2]), "r"(w[4 * pc + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ds);
      // a finished dV/dK chain (more pairs follow): into the accumulators before
      // these warpgroups hand over the next P^T, whose dV starts a new chain
      if ((i + 1) % kChain == 0 && i + 1 < npairs) {
        if (!wait_warp(b_dsf, pi, 253)) { ok = false; break; }
        tc_fence_after();
        flush_dkdv();
        tc_fence_before();
      }
    }
    // every MMA of the CTA is done once dK and dQ^T of the last pair are
    if (ok && npairs > 0 && wait_warp(b_dsf, (uint32_t)(npairs - 1) & 1u, 254)) {
      tc_fence_after();
      flush_dkdv();
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;");
    // ------------------------------------------------------------ dQ warpgroup
    // TMEM lanes = the half's 128 columns (this warp: 32 of them), 64 query
    // columns.  Each warp stages 32 query rows x its 32 columns (128-byte
    // swizzle, the accumulator map's box) and adds them with a bulk tensor
    // reduction, twice per pair.  Query rows outside the range carry exact
    // zeros (their dS columns are masked); rows past T are clipped by the map.
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t aQ = tmem_addr(tmem, lane_base, tQ);
    const uint32_t wbuf = sStg + (uint32_t)(warp & 3) * 4096;
    const bool lead = lane == 0;
    const int col = 128 * half + (int)lane_base;  // first accumulator column of this warp
    for (int j = 0; j < npairs; ++j) {
      if (!wait_warp(b_dq, (uint32_t)j & 1u, 260)) break;
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(aQ, r[0]);
      tmem_ld32(aQ + 32, r[1]);
      tmem_ld_wait();
      reg_fence32(r[0]);
      reg_fence32(r[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_dqf);  // dQ^T has left tensor memory
#pragma unroll
      for (int rd = 0; rd < 2; ++rd) {
        if (lead) bulk_wait_read();  // the buffer's previous box has been read
        __syncwarp();
        // row q of the box = query q0 + 32 rd + q; this lane's column sits in
        // 16-byte chunk (lane / 4) ^ (q % 8) of the row
#pragma unroll
        for (int q = 0; q < 32; ++q)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(wbuf + (uint32_t)q * 128 +
                                                       ((uint32_t)((lane >> 2) ^ (q & 7)) << 4) + (lane & 3) * 4),
                       "f"(__uint_as_float(r[rd][q]))
                       : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lead) {
          tma_reduce_add_3d(&tmDQ, wbuf, col, pl.head(j), pl.start(j) + 32 * rd);
          bulk_commit();
        }
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

}  // namespace

cudaError_t launch_bwd_step_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tl, const CUtensorMap& td,
                                 const CUtensorMap& tdq, const BwdParams& p, int num_items, cudaStream_t stream) {
  auto kern = ring_bwd_d256_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, b256::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = 2LL * num_items;  // two column halves per work item
  if (grid <= 0) return cudaSuccess;
  BwdParams q = p;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  q.next_cta = sms;
  kern<<<(unsigned)grid, 512, b256::kSmem, stream>>>(tq, tk, tv, tdo, tl, td, tdq, q);
  return cudaGetLastError();
}

}  // namespace ra
