// fwd.cu -- one ring step of the forward pass on tcgen05 tensor cores.
//
// One CTA takes up to 256 query rows (two 128-row tiles Q0, Q1) of one head and
// runs the online softmax over the key/value tiles of the shard its query
// shard holds at this ring step (NVSHMEM/XLA page, "Paralelismo de contexto y
// atencion en anillo": attention is computed incrementally as KV blocks
// circulate).  The step's partial (O_s, LSE_s) is merged exactly into the
// running (O, LSE) in the epilogue (the Accelerate guide's `combine`, read as
// the log-sum-exp merge).
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q0/Q1 once, then K_j, V_j into a ring of stages
//   warp 1      TMEM owner + UMMA issuer for Q0
//   warp 2      UMMA issuer for Q1
//   warps 4-7   softmax / correction / epilogue of Q0 (TMEM lanes 0-127)
//   warps 8-11  softmax / correction / epilogue of Q1
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 and O1 after that.
// P (bf16) overwrites the first 64 columns of S and feeds the P.V MMA straight
// from tensor memory.  Each Q tile's issuer runs PV(j) then S(j+1); the two
// softmax warpgroups take turns, so one tile's softmax overlaps the other
// tile's MMAs.
// Epilogue traffic: each warp passes its 32 rows through its slice of its Q
// tile's shared-memory buffer (idle once the tile's last QK is done), so every
// global load and store of the running (or final) output covers whole rows.
// The producer prefetches into L2 the Q tiles of the CTA that will follow
// this one on the SM.
#include "ring_attn_internal.h"
#include "tc.cuh"

namespace ra {
namespace {

#define kNegInf (-__int_as_float(0x7f800000))
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: after a max update P stays below 2^8
// A tile computed against the running reference is kept while its row sum of
// P stays at or below this bound (so every P <= 2^16; fp32 accumulators and
// bf16 P have room to spare).
constexpr float kSpecSumLimit = 65536.0f;

template <int D, bool kFused>
struct FwdCfg {
  static constexpr int kTile = 128 * D * 2;  // bytes of one 128-row bf16 tile
  // K/V stages: a fifth stage at d = 128 fits in shared memory (225.5 KB) and
  // helps the single launch (1250 -> 1262 TFLOP/s at 128K) but not the
  // ring-step launches (1195 -> 1181), whose CTAs are short.
  static constexpr int kStages = D == 128 ? (kFused ? 5 : 4) : 8;
  static constexpr int kQBytes = 2 * kTile;
  static constexpr int kKVBytes = kStages * kTile;
  static constexpr int kBarOff = kQBytes + kKVBytes;
  static constexpr int kSmem = kBarOff + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
};

// Key tiles of one CTA.  Ring-step launch: up to two sorted key ranges, cut
// into 128-key tiles.  Single launch over the ring: an explicit table of
// (tile start, range end), ring step by ring step.
template <bool kFused>
struct TileList {
  int32_t kb0, ke0, kb1, ke1, n0, n;
  const int2* tab;
  __device__ __forceinline__ int start(int j) const {
    if constexpr (kFused) return tab[j].x;
    else return j < n0 ? kb0 + 128 * j : kb1 + 128 * (j - n0);
  }
  __device__ __forceinline__ int end(int j) const {
    if constexpr (kFused) return tab[j].y;
    else return j < n0 ? ke0 : ke1;
  }
};

__device__ __forceinline__ int ceil128(int a, int b) { return b > a ? (b - a + 127) / 128 : 0; }

template <int D, bool kFused>
__global__ void __launch_bounds__(384, 1)
    ring_fwd_step_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D, kFused>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + C::kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  // barrier map
  const uint32_t b_q = smem_u32(bars + 0);
  const uint32_t b_full = smem_u32(bars + 1);                      // [kStages]
  const uint32_t b_empty = smem_u32(bars + 1 + C::kStages);        // [kStages]
  const uint32_t b_s = smem_u32(bars + 1 + 2 * C::kStages);        // [2] S ready / O final
  const uint32_t b_p = smem_u32(bars + 3 + 2 * C::kStages);        // [2] P written
  const uint32_t b_drain = smem_u32(bars + 5 + 2 * C::kStages);    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7 + 2 * C::kStages);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  // A CTA of this grid already gave up: do no work (fail fast, no waits).
  if (*reinterpret_cast<volatile int*>(p.status) != 0) return;
  // Ring-step launches: the next step may start on the SMs this grid frees;
  // it reads the running (O, LSE) only after this grid has completed.
  if constexpr (!kFused) pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const FwdItem it = p.items[blockIdx.x / p.Hq];

  TileList<kFused> tl;
  int n_act[2];   // key tiles each Q tile sees
  bool q_act[2];
  int last_row[2];
#pragma unroll
  for (int qt = 0; qt < 2; ++qt) {
    const int first = it.q0 + 128 * qt;
    q_act[qt] = first < it.q1;
    last_row[qt] = min(first + 128, it.q1) - 1;
  }
  if constexpr (kFused) {
    tl.tab = p.tiles + it.kb0;
    tl.n = it.ke0;
    n_act[0] = q_act[0] ? it.kb1 : 0;
    n_act[1] = q_act[1] ? it.ke1 : 0;
  } else {
    tl.kb0 = it.kb0; tl.ke0 = it.ke0; tl.kb1 = it.kb1; tl.ke1 = it.ke1;
    tl.n0 = ceil128(it.kb0, it.ke0);
    tl.n = tl.n0 + ceil128(it.kb1, it.ke1);
    // here the active key tiles of each Q tile form a prefix of the tile list
#pragma unroll
    for (int qt = 0; qt < 2; ++qt) {
      int n = 0;
      if (q_act[qt]) {
        if (!p.causal) n = tl.n;
        else while (n < tl.n && tl.start(n) <= last_row[qt]) ++n;
      }
      n_act[qt] = n;
    }
  }
  // does a Q tile (in scalars, so the arrays above stay in registers) see key
  // tile j; causal: a tile that starts after its last row is skipped
  auto active = [&](int j, bool qa, int last, int na) -> bool {
    if constexpr (kFused) return qa && (!p.causal || tl.start(j) <= last);
    else return j < na;
  };

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 2);  // one commit per MMA issuer
    }
    mbar_init(b_s, 1); mbar_init(b_s + 8, 1);
    mbar_init(b_p, 4); mbar_init(b_p + 8, 4);  // one arrival per softmax warp
    mbar_init(b_drain, 1); mbar_init(b_drain + 8, 1);
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

  // Register split: 384 threads x 168 at launch.  The producer/MMA warpgroup
  // drops to 56 and the two softmax warpgroups rise to 216:
  // 128 x 56 + 256 x 216 = 62464 <= 64512.  Each warpgroup sets its limit at
  // the head of its own branch, so no code is shared across the two limits.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV);
      mbar_expect_tx(b_q, (q_act[0] ? C::kTile : 0) + (q_act[1] ? C::kTile : 0));
      for (int qt = 0; qt < 2; ++qt) {
        if (!q_act[qt]) continue;
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_3d(sQ + qt * C::kTile + hf * 16384, &tmQ, b_q, 64 * hf, h, it.q0 + 128 * qt);
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < tl.n && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind) {
          const int st = issued % C::kStages;
          const uint32_t ph = (issued / C::kStages) & 1;
          if (!mbar_wait(b_empty + 8 * st, ph ^ 1, ab, 101)) { ok = false; break; }
          mbar_expect_tx(b_full + 8 * st, C::kTile);
          const CUtensorMap* m = kind == 0 ? &tmK : &tmV;
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_3d(sKV + st * C::kTile + hf * 16384, m, b_full + 8 * st, 64 * hf, g, tl.start(j));
          ++issued;
        }
      }
      if constexpr (!kFused) {
        // CTAs run one per SM and start in order, so CTA b + next_cta takes an
        // SM about when this one ends: bring its Q tiles into L2 now, so its
        // first QK waits on L2 rather than on HBM.
        const long long nb = (long long)blockIdx.x + p.next_cta;
        if (ok && p.next_cta > 0 && nb < (long long)gridDim.x) {
          const FwdItem nx = p.items[nb / p.Hq];
          const int nh = (int)(nb % p.Hq);
          for (int qt = 0; qt < 2; ++qt) {
            const int first = nx.q0 + 128 * qt;
            if (first >= nx.q1) continue;
            for (int hf = 0; hf < D / 64; ++hf) tma_prefetch_l2_3d(&tmQ, 64 * hf, nh, first);
          }
          // and its first key/value tile
          const bool r0 = ceil128(nx.kb0, nx.ke0) > 0;
          if (r0 || ceil128(nx.kb1, nx.ke1) > 0) {
            const int nk0 = r0 ? nx.kb0 : nx.kb1;
            const int ng = nh / (p.Hq / p.Hkv);
            for (int hf = 0; hf < D / 64; ++hf) {
              tma_prefetch_l2_3d(&tmK, 64 * hf, ng, nk0);
              tma_prefetch_l2_3d(&tmV, 64 * hf, ng, nk0);
            }
          }
        }
      }
      if (!ok) {  // drain this CTA's copies still in flight
        mbar_wait_drain(b_q, 0);
        for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
          mbar_wait_drain(b_full + 8 * (i % C::kStages), (i / C::kStages) & 1);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per Q tile.  A thread that has issued tcgen05.mma and
    // then waits on a barrier is held until the tensor pipe has taken its MMAs,
    // so with a single issuer the pipe runs dry on every wait; with two, one
    // tile's MMAs keep it busy while the other issuer waits.  Both issuers walk
    // every K/V stage in order (waiting for it to be full, then committing its
    // release), so each stage release gets exactly one arrival from each.
    const int qt = warp - 1;
    if (lane == 0) {
      const int na = qt == 0 ? n_act[0] : n_act[1];
      const bool my_qa = qt == 0 ? q_act[0] : q_act[1];
      const int my_last = qt == 0 ? last_row[0] : last_row[1];
      auto act = [&](int j) { return active(j, my_qa, my_last, na); };
      const uint32_t tS = tmem + qt * 128, tO = tmem + 256 + qt * D;
      bool ok = mbar_wait(b_q, 0, ab, 102);
      tc_fence_after();
      int stage = 0;
      uint32_t kph = 0;
      auto advance = [&]() { if (++stage == C::kStages) { stage = 0; kph ^= 1; } };
      // Every operand descriptor is the shared-memory base's plus constants
      // (sdesc_at), so each MMA costs an add or two to issue.
      const uint64_t d0 = sdesc_sw128(sQ, 0, 1024);
      auto qk = [&](int kst) {
        const uint64_t b = opaque(d0);
        const uint64_t dq = sdesc_at(b, (uint32_t)qt * C::kTile, 0);
        const uint64_t dk = sdesc_at(b, (uint32_t)(C::kQBytes + kst * C::kTile), 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_ss(tS, sdesc_at(dq, off, 16), sdesc_at(dk, off, 16), C::kIdescQK, kk > 0);
        }
      };
      // b_s is committed right after each QK of a tile this Q tile sees (S
      // ready; it also covers the P.V before it), and once more after the last
      // P.V (O final)
      if (ok) ok = mbar_wait(b_full + 8 * stage, kph, ab, 103);
      if (ok) {
        tc_fence_after();
        if (act(0)) { qk(stage); umma_commit(b_s + 8 * qt); }
        umma_commit(b_empty + 8 * stage);
        advance();
      }
      uint32_t pph = 0;
      int u = 0;  // P.V issued so far
      for (int j = 0; j < tl.n && ok; ++j) {
        const int vst = stage;
        if (!mbar_wait(b_full + 8 * vst, kph, ab, 104)) { ok = false; break; }
        tc_fence_after();
        advance();  // stage now holds K_{j+1}
        if (act(j)) {
          if (!mbar_wait(b_p + 8 * qt, pph, ab, 105)) { ok = false; break; }
          pph ^= 1;
          tc_fence_after();
          const uint64_t dv = sdesc_at(opaque(d0), (uint32_t)(C::kQBytes + vst * C::kTile), 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tO, tS + kk * 8, sdesc_at(dv, kk * 2048, 16384), C::kIdescPV, (u > 0 || kk > 0) ? 1u : 0u);
          if (++u == na) umma_commit(b_s + 8 * qt);  // O final
        }
        umma_commit(b_empty + 8 * vst);  // V_j: free once this tile's P.V has run
        if (j + 1 < tl.n) {
          if (!mbar_wait(b_full + 8 * stage, kph, ab, 106)) { ok = false; break; }
          tc_fence_after();
          if (act(j + 1)) { qk(stage); umma_commit(b_s + 8 * qt); }  // S(j+1) ready
          umma_commit(b_empty + 8 * stage);  // K_{j+1}: free once this tile's QK has run
          advance();
        }
      }
      if (!ok) {  // let issued MMAs finish before tensor memory is released
        umma_commit(b_drain + 8 * qt);
        mbar_wait_drain(b_drain + 8 * qt, 0);
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
    // ------------------------------------------------------------ softmax
    const int qt = (warp - 4) >> 2;
    const int tid = threadIdx.x - 128 * (1 + qt);
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t tS = tmem_addr(tmem, lane_base, qt * 128);
    const uint32_t tO = tmem_addr(tmem, lane_base, 256 + qt * D);
    const int row0 = it.q0 + 128 * qt;
    const int row = row0 + tid;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    float m_ref = kNegInf, l_sum = 0.f, l_rnd = 0.f;
    uint32_t sph = 0;
    bool ok = true;
    const int na = qt == 0 ? n_act[0] : n_act[1];
    const bool qa = qt == 0 ? q_act[0] : q_act[1];
    const int na_other = qt == 0 ? n_act[1] : n_act[0];
    const int my_last = qt == 0 ? last_row[0] : last_row[1];
    int u = 0;  // tiles done so far
    for (int j = 0; j < tl.n; ++j) {
      if (!active(j, qa, my_last, na)) continue;
      if (!kFused && u == na - 1 && row < it.q1 && !(it.flags & kFirstStep)) {
        // last tile: bring this row's running (O, LSE) towards L2 for the merge
        const char* orow = reinterpret_cast<const char*>(p.o_run + ((size_t)row * p.Hq + h) * D);
#pragma unroll
        for (int c = 0; c < D * 4; c += 128) prefetch_l2(orow + c);
        prefetch_l2(p.lse + (size_t)h * p.T + row);
      }
      if (!mbar_wait(b_s + 8 * qt, sph, ab, 110)) { ok = false; break; }
      sph ^= 1;
      tc_fence_after();
      uint32_t r[4][32];
      tmem_ld32(tS + 0, r[0]);
      tmem_ld32(tS + 32, r[1]);
      tmem_ld32(tS + 64, r[2]);
      tmem_ld32(tS + 96, r[3]);
      // The two softmax warpgroups take turns (Q0 tile j after Q1 tile j-1, Q1
      // tile j after Q0 tile j): each then runs alone on the SM's schedulers,
      // and their MMAs reach the tensor pipe interleaved instead of together.
      const int k_other = u - (qt == 0 ? 1 : 0);
      const bool turn = k_other < 0 || k_other >= na_other ||
                        mbar_wait(b_p + 8 * (1 - qt), (uint32_t)k_other & 1u, ab, 112);
      tmem_ld_wait();
      if (!turn) { ok = false; break; }
      reg_fence32(r[0]); reg_fence32(r[1]); reg_fence32(r[2]); reg_fence32(r[3]);
      const int kst = tl.start(j), kend = tl.end(j);
      const bool need_mask = (kst + 128 > kend) || (p.causal && kst + 127 > row0);
      if (need_mask) {
        const int lim = p.causal ? min(kend - 1, row) : kend - 1;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (kst + c > lim) r[c >> 5][c & 31] = __float_as_uint(kNegInf);
      }
      // Two row sums: of P (for the LSE) and of the bf16-rounded P that the PV MMA
      // consumes (to normalise O, so O stays an exact convex combination of V).
      // Scale-and-shift and the exact sum run on packed fp32 pairs; the rounded
      // sum adds the bf16 halves straight into fp32.
      uint64_t nm2 = 0, ls_a = 0, ls_b = 0;
      float lr0 = 0.f, lr1 = 0.f, lr2 = 0.f, lr3 = 0.f;
      auto p_chunk = [&](int c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t x =
              f2_fma(f2_pack(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), sl2x2, nm2);
          float x0, x1;
          f2_unpack(x, x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          pk[i] = pack_bf16x2(p0, p1);
          if (i & 1) {
            ls_b = f2_add(ls_b, f2_pack(p0, p1));
            add_bf16x2_to(lr2, lr3, pk[i]);
          } else {
            ls_a = f2_add(ls_a, f2_pack(p0, p1));
            add_bf16x2_to(lr0, lr1, pk[i]);
          }
        }
        tmem_st16(tS + 16 * c, pk);
      };
      // P = 2^(S log2e scale - m) for the whole tile, written over S in TMEM
      auto p_tile = [&](float m_use) {
        nm2 = f2_pack(-m_use, -m_use);
        ls_a = ls_b = 0;
        lr0 = lr1 = lr2 = lr3 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) p_chunk(c);
      };
      auto tile_sum = [&]() {
        float a0, a1, b0, b1;
        f2_unpack(ls_a, a0, a1);
        f2_unpack(ls_b, b0, b1);
        return (a0 + a1) + (b0 + b1);
      };
      // First try the running reference max as it stands, without looking at
      // this tile's max: that stands unless the tile's P would grow too large,
      // which is rare once the first tile has set the reference.  Otherwise (and
      // for a warp with a row that has seen no key yet) take the row max, move
      // the reference when it grew past the threshold, and redo the tile.  One
      // copy of the tile code serves both passes (instruction-cache footprint).
      bool exact = __any_sync(0xffffffffu, m_ref == kNegInf);
      bool rescale = false;
      float alpha = 1.f;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (exact) {
          // row max: eight independent chains of three-input max, eight deep
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = kNegInf;
#pragma unroll
          for (int i = 0; i < 16; i += 2)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx[k] = fmax3(mx[k], __uint_as_float(r[k >> 1][16 * (k & 1) + i]),
                            __uint_as_float(r[k >> 1][16 * (k & 1) + i + 1]));
          const float m_tile =
              fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7]))) * sl2;
          const float m_new = fmaxf(m_ref, m_tile);
          rescale = m_new > m_ref + kRescaleThreshold;
          if (rescale) {
            // The reference max is kept integral (log2 units): partials over any
            // split of the keys then differ by exact powers of two, so the bf16
            // rounding of P does not depend on the ring layout.
            const float m_int = ceilf(m_new);
            alpha = ex2_approx(m_ref - m_int);
            l_sum *= alpha;
            l_rnd *= alpha;
            m_ref = m_int;
          }
        }
        p_tile((m_ref == kNegInf) ? 0.f : m_ref);
        if (exact || !__any_sync(0xffffffffu, !(tile_sum() <= kSpecSumLimit))) break;
        tmem_st_wait();  // the redo overwrites these P stores
        exact = true;
      }
      if (u > 0 && __any_sync(0xffffffffu, rescale)) {
        // O holds PV of the tiles before (complete: this S was committed after
        // their P.V), and must be rescaled before this tile's P.V adds to it.
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait();
          reg_fence32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + 32 * c, o);
        }
      }
      // One arrival per warp: the shared-memory unit takes an mbarrier's
      // arrivals one at a time, so 128 of them would hold the MMA issuer back.
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p + 8 * qt);
      l_sum += tile_sum();
      l_rnd += (lr0 + lr1) + (lr2 + lr3);
      ++u;
    }
    // the epilogue exchanges values between lanes: the whole warp takes it or
    // skips it (a wait that gave up in any lane has already raised the abort)
    ok = __all_sync(0xffffffffu, ok);
    if (ok && qa && (na > 0 || (it.flags & kFirstStep))) {
      if constexpr (kFused) {
        if (na > 0) {
          ok = mbar_wait(b_s + 8 * qt, sph, ab, 111);  // O final
          tc_fence_after();
        }
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok && kFused) {
        // the whole ring is done: O = (sum of P V) / (sum of the bf16 P), final LSE
        const bool valid = row < it.q1;
        const float lse_b = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) * kLn2 : kNegInf;
        const float inv_l = (l_rnd > 0.f) ? 1.f / l_rnd : 0.f;
        if (valid) p.lse[(size_t)h * p.T + row] = lse_b;
        // rows leave through this warp's slice of its Q tile's buffer, so each
        // store instruction covers whole rows (as in the ring-step merge below)
        constexpr int kHalf = D / 2;
        constexpr int kChunks = kHalf / 4;
        constexpr int kPer = 32 / kChunks;
        constexpr int kSteps = 32 / kPer;
        const uint32_t scratch = sQ + qt * C::kTile + (uint32_t)(warp & 3) * (C::kTile / 4);
        const int sub = lane / kChunks, ch = lane % kChunks;
        const int wrow0 = row0 + (int)lane_base;
        const size_t obase = ((size_t)wrow0 * p.Hq + h) * D + 4 * ch;
        const size_t rstride = (size_t)p.Hq * D;
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
#pragma unroll
          for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t o[32];
            if (na > 0) {
              tmem_ld32(tO + ps * kHalf + 32 * c, o);
              tmem_ld_wait();
              reg_fence32(o);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int kc = 8 * c + k;
              const uint32_t addr = scratch + (uint32_t)lane * (kHalf * 4) + (uint32_t)((kc ^ (lane % kChunks)) << 4);
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                           "f"(__uint_as_float(o[4 * k]) * inv_l), "f"(__uint_as_float(o[4 * k + 1]) * inv_l),
                           "f"(__uint_as_float(o[4 * k + 2]) * inv_l), "f"(__uint_as_float(o[4 * k + 3]) * inv_l)
                           : "memory");
            }
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int rr = kPer * i + sub;
            float4 v;
            const uint32_t addr = scratch + (uint32_t)rr * (kHalf * 4) + (uint32_t)((ch ^ (rr % kChunks)) << 4);
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
            if (wrow0 + rr >= it.q1) continue;
            const size_t off = obase + rr * rstride + ps * kHalf;
            if (p.o_bf16)
              *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.o_out) + off) =
                  make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
            else
              *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o_out) + off) = v;
          }
          __syncwarp();
        }
      } else if (ok) {
        pdl_wait();  // the previous ring step's (O, LSE) are complete and visible
        const bool valid = row < it.q1;
        const bool first = (it.flags & kFirstStep) != 0;
        const float lse_b = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) * kLn2 : kNegInf;
        const float inv_l = (l_rnd > 0.f) ? 1.f / l_rnd : 0.f;
        float* lse_ptr = p.lse + (size_t)h * p.T + row;
        const float lse_a = (valid && !first) ? *lse_ptr : kNegInf;
        float wa = 0.f, wb = 1.f, lse_new = lse_b;
        if (lse_b == kNegInf) { wa = 1.f; wb = 0.f; lse_new = lse_a; }
        else if (lse_a != kNegInf) {
          const float a2 = lse_a * 1.4426950408889634f, b2 = lse_b * 1.4426950408889634f;
          const float mx = fmaxf(a2, b2);
          const float n2 = mx + log2f(1.f + exp2f(-fabsf(a2 - b2)));
          wa = exp2f(a2 - n2);
          wb = exp2f(b2 - n2);
          lse_new = n2 * kLn2;
        }
        wb *= inv_l;
        const bool write = valid && (first || lse_b != kNegInf);
        const bool read_old = valid && !first && lse_a != kNegInf && lse_b != kNegInf;
        // The running rows are read and written whole, through this warp's
        // slice of its Q tile's buffer (free: the tile's last QK is done):
        // the thread of a row writes its columns there, then every load and
        // store instruction covers kPer full rows (16 bytes per lane), instead
        // of 16 bytes of 32 different rows.  Two passes of D/2 columns.
        constexpr int kHalf = D / 2;          // columns per pass
        constexpr int kChunks = kHalf / 4;    // 16-byte chunks of a row per pass
        constexpr int kPer = 32 / kChunks;    // rows per instruction
        constexpr int kSteps = 32 / kPer;     // instructions per pass
        const uint32_t scratch = sQ + qt * C::kTile + (uint32_t)(warp & 3) * (C::kTile / 4);
        const int sub = lane / kChunks, ch = lane % kChunks;
        const int wrow0 = row0 + (int)lane_base;  // the warp's first row
        float* obase = p.o_run + ((size_t)wrow0 * p.Hq + h) * D + 4 * ch;
        const size_t rstride = (size_t)p.Hq * D;
        // A pass's loads of the old rows go out together (one round trip; the
        // rows were hinted into L2 during the last key tile).  The first
        // pass's go out before the wait for the final O: they need only the
        // previous ring step.
        float4 old[kSteps];
        auto load_old = [&](int ps) {
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int rr = kPer * i + sub;
            const bool ro = __shfl_sync(0xffffffffu, read_old, rr) != 0;
            old[i] = ro ? *reinterpret_cast<const float4*>(obase + rr * rstride + ps * kHalf)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        };
        load_old(0);
        if (na > 0) {
          ok = mbar_wait(b_s + 8 * qt, sph, ab, 111);  // O final
          tc_fence_after();
        }
        ok = __all_sync(0xffffffffu, ok);
#pragma unroll
        for (int ps = 0; ps < 2 && ok; ++ps) {
          if (ps > 0) load_old(ps);
#pragma unroll
          for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t o[32];
            if (na > 0) {
              tmem_ld32(tO + ps * kHalf + 32 * c, o);
              tmem_ld_wait();
              reg_fence32(o);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int kc = 8 * c + k;  // chunk within the pass
              const uint32_t addr = scratch + (uint32_t)lane * (kHalf * 4) + (uint32_t)((kc ^ (lane % kChunks)) << 4);
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                           "f"(__uint_as_float(o[4 * k]) * wb), "f"(__uint_as_float(o[4 * k + 1]) * wb),
                           "f"(__uint_as_float(o[4 * k + 2]) * wb), "f"(__uint_as_float(o[4 * k + 3]) * wb)
                           : "memory");
            }
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int rr = kPer * i + sub;
            const float w = __shfl_sync(0xffffffffu, wa, rr);
            const bool ro = __shfl_sync(0xffffffffu, read_old, rr) != 0;
            const bool wr = __shfl_sync(0xffffffffu, write, rr) != 0;
            float4 v;
            const uint32_t addr = scratch + (uint32_t)rr * (kHalf * 4) + (uint32_t)((ch ^ (rr % kChunks)) << 4);
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
            if (ro) {
              const float4 u = old[i];
              v.x = fmaf(w, u.x, v.x);
              v.y = fmaf(w, u.y, v.y);
              v.z = fmaf(w, u.z, v.z);
              v.w = fmaf(w, u.w, v.w);
            }
            if (wr) *reinterpret_cast<float4*>(obase + rr * rstride + ps * kHalf) = v;
          }
          __syncwarp();  // the next pass reuses the slice
        }
        if (ok && write) *lse_ptr = lse_new;
      }
    }
  }

  // keep the launches' completion order: this grid completes after the previous one
  if (!kFused && threadIdx.x == 0 && blockIdx.x == gridDim.x - 1) pdl_wait();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kFused>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                   int num_items, cudaStream_t stream) {
  auto kern = ring_fwd_step_kernel<D, kFused>;
  constexpr int kSmem = FwdCfg<D, kFused>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)num_items * p.Hq;
  if (grid <= 0) return cudaSuccess;
  FwdParams q = p;
  if (!kFused) {  // one CTA per SM (shared memory): the stride to the CTA that follows on an SM
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    q.next_cta = sms;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kFused ? 0 : 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, q);
}

}  // namespace

cudaError_t launch_fwd_step(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, int num_items, cudaStream_t stream) {
  if (head_dim == 128) return launch<128, false>(tq, tk, tv, p, num_items, stream);
  if (head_dim == 64) return launch<64, false>(tq, tk, tv, p, num_items, stream);
  if (head_dim == 256) return launch_fwd_step_d256(tq, tk, tv, p, num_items, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_fused(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int num_items, cudaStream_t stream) {
  if (head_dim == 128) return launch<128, true>(tq, tk, tv, p, num_items, stream);
  if (head_dim == 64) return launch<64, true>(tq, tk, tv, p, num_items, stream);
  if (head_dim == 256) return launch_fwd_fused_d256(tq, tk, tv, p, num_items, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ra
