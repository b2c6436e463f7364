// fwd256.cu -- the forward for head_dim 256 on tcgen05 tensor cores: one ring
// step per launch (running (O, LSE) merged in the epilogue), or the whole ring
// in one launch (running state kept on chip).
//
// At head_dim 256 one output accumulator takes 256 tensor-memory columns, so a
// CTA holds one 128-row query tile: S is double-buffered (two 128-column
// buffers) and O takes the other 256 columns.  While the softmax warpgroup
// works on S(j), the tensor pipe computes S(j+1) into the other buffer.  K and
// V tiles (128 rows x 256 columns, 64 KB each) move through a ring of five
// 32 KB half-tile stages, loaded in the order the MMAs consume them:
// K(0), then K(j+1), V(j) for every j.  The tensor work per key tile (S and
// P.V, 2 x 128 x 128 x 256 multiply-adds) is twice that of head_dim 128, so
// one softmax warpgroup keeps up with one Q tile.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q once, then the K/V half tiles
//   warp 1      TMEM owner + UMMA issuer: S(0), then S(j+1) and P(j).V(j)
//   warps 4-7   softmax / correction / epilogue (TMEM lanes 0-127 = rows)
// P (bf16) overwrites the first 64 columns of its S buffer and feeds the P.V
// MMA straight from tensor memory; O is rescaled in tensor memory when the
// reference maximum moves (after P(j-1).V(j-1) has completed).
#include "ring_attn_internal.h"
#include "tc.cuh"

namespace ra {
namespace {

#define kNegInf256 (-__int_as_float(0x7f800000))
constexpr float kLn2_256 = 0.69314718055994530942f;
constexpr float kRescaleThreshold256 = 8.0f;  // log2 units (see the head_dim 64/128 kernel)
constexpr float kSpecSumLimit256 = 65536.0f;

constexpr int kD = 256;
constexpr int kQBytes = 128 * kD * 2;   // 64 KB: four 64-column boxes
constexpr int kHalfTile = 128 * 128 * 2;  // 32 KB: a K or V tile's 128 columns
constexpr int kStages = 5;
constexpr int kBarOff = kQBytes + kStages * kHalfTile;
constexpr int kSmem = kBarOff + 256 + 1024;  // barriers + alignment slack
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);  // N = 128: one half of O

// The t-th tile of the load/consume order over n key tiles: K(0), then
// K(j+1) (while j + 1 < n) and V(j) for j = 0 .. n-1.
__device__ __forceinline__ void seq_tile(int t, int n, bool& is_v, int& j) {
  if (t == 0) {
    is_v = false;
    j = 0;
    return;
  }
  const int u = t - 1;
  if (u < 2 * (n - 1)) {
    is_v = (u & 1) != 0;
    j = is_v ? (u >> 1) : (u >> 1) + 1;
  } else {
    is_v = true;
    j = n - 1;
  }
}

template <bool kFused>
struct Tiles256 {
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

__device__ __forceinline__ int tiles_of(int a, int b) { return b > a ? (b - a + 127) / 128 : 0; }

template <bool kFused>
__global__ void __launch_bounds__(256, 1)
    ring_fwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const uint32_t b_q = smem_u32(bars + 0);
  const uint32_t b_full = smem_u32(bars + 1);                 // [kStages]
  const uint32_t b_empty = smem_u32(bars + 1 + kStages);      // [kStages]
  const uint32_t b_s = smem_u32(bars + 1 + 2 * kStages);      // [2] S(j) ready, per buffer
  const uint32_t b_p = smem_u32(bars + 3 + 2 * kStages);      // P(j) written
  const uint32_t b_o = smem_u32(bars + 4 + 2 * kStages);      // P(j).V(j) done
  const uint32_t b_drain = smem_u32(bars + 5 + 2 * kStages);
  // O final: committed once, after the last P.V.  (b_o cannot serve: when the
  // softmax finishes its last tile, the P.V of the tile before it may still be
  // running, and a parity wait cannot tell three phase counts apart.)
  const uint32_t b_of = smem_u32(bars + 6 + 2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7 + 2 * kStages);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  if (*reinterpret_cast<volatile int*>(p.status) != 0) return;
  if constexpr (!kFused) pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const FwdItem it = p.items[blockIdx.x / p.Hq];

  // one query tile of up to 128 rows; every key tile of the list is active
  // for it (the planner clips key ranges to keys < q1, and q1 - q0 <= 128)
  Tiles256<kFused> tl;
  if constexpr (kFused) {
    tl.tab = p.tiles + it.kb0;
    tl.n = it.ke0;
  } else {
    tl.kb0 = it.kb0; tl.ke0 = it.ke0; tl.kb1 = it.kb1; tl.ke1 = it.ke1;
    tl.n0 = tiles_of(it.kb0, it.ke0);
    tl.n = tl.n0 + tiles_of(it.kb1, it.ke1);
  }
  const int n = tl.n;
  const int row0 = it.q0;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    mbar_init(b_s, 1); mbar_init(b_s + 8, 1);
    mbar_init(b_p, 4);  // one arrival per softmax warp
    mbar_init(b_o, 1);
    mbar_init(b_drain, 1);
    mbar_init(b_of, 1);
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
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV);
      bool ok = true;
      int issued = 0;
      if (n > 0) {
        mbar_expect_tx(b_q, kQBytes);
        for (int b = 0; b < 4; ++b) tma_load_3d(sQ + b * 16384, &tmQ, b_q, 64 * b, h, row0);
        for (int t = 0; t < 2 * n && ok; ++t) {
          bool is_v;
          int j;
          seq_tile(t, n, is_v, j);
          const CUtensorMap* m = is_v ? &tmV : &tmK;
          for (int half = 0; half < 2; ++half) {
            const int st = issued % kStages;
            const uint32_t ph = (issued / kStages) & 1;
            if (!mbar_wait(b_empty + 8 * st, ph ^ 1, ab, 131)) { ok = false; break; }
            mbar_expect_tx(b_full + 8 * st, kHalfTile);
            for (int b = 0; b < 2; ++b)
              tma_load_3d(sKV + st * kHalfTile + b * 16384, m, b_full + 8 * st, 128 * half + 64 * b, g,
                          tl.start(j));
            ++issued;
          }
        }
      }
      if constexpr (!kFused) {
        // CTA b + next_cta takes this SM about when this one ends: its Q tile to L2
        const long long nb = (long long)blockIdx.x + p.next_cta;
        if (ok && p.next_cta > 0 && nb < (long long)gridDim.x) {
          const FwdItem nx = p.items[nb / p.Hq];
          const int nh = (int)(nb % p.Hq);
          for (int b = 0; b < 4; ++b) tma_prefetch_l2_3d(&tmQ, 64 * b, nh, nx.q0);
        }
      }
      if (!ok) {  // drain this CTA's copies still in flight
        if (n > 0) mbar_wait_drain(b_q, 0);
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
          mbar_wait_drain(b_full + 8 * (i % kStages), (i / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      bool ok = mbar_wait(b_q, 0, ab, 132);
      tc_fence_after();
      int c = 0;  // half tiles consumed so far (same order as loaded)
      auto wait_full = [&](int idx) -> bool {
        return mbar_wait(b_full + 8 * (idx % kStages), (idx / kStages) & 1, ab, 133);
      };
      // S(j) = Q K(j)^T into buffer j & 1
      // Every operand descriptor is the shared-memory base's plus constants
      // (sdesc_at), so each MMA costs an add or two to issue.
      const uint64_t d0 = sdesc_sw128(sQ, 0, 1024);
      auto qk = [&](int j) -> bool {
        const uint32_t tS = tmem + (uint32_t)(j & 1) * 128;
        for (int half = 0; half < 2; ++half) {
          if (!wait_full(c)) return false;
          tc_fence_after();
          const uint64_t b = opaque(d0);
          const uint64_t dk = sdesc_at(b, (uint32_t)(kQBytes + (c % kStages) * kHalfTile), 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int gk = 8 * half + kk;  // K step over the 256 columns of Q
            const uint32_t qoff = (gk >> 2) * 16384 + (gk & 3) * 32;
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_ss(tS, sdesc_at(b, qoff, 16), sdesc_at(dk, koff, 16), kIdescQK, (half | kk) ? 1u : 0u);
          }
          umma_commit(b_empty + 8 * (c % kStages));  // the half tile is free once these MMAs ran
          ++c;
        }
        umma_commit(b_s + 8 * (j & 1));
        return true;
      };
      // O += P(j) V(j): P from tensor memory (first 64 columns of S(j)'s
      // buffer), one MMA group per 128-column half of V and O
      auto pv = [&](int j) -> bool {
        const uint32_t tS = tmem + (uint32_t)(j & 1) * 128;
        for (int half = 0; half < 2; ++half) {
          if (!wait_full(c)) return false;
          tc_fence_after();
          const uint64_t dv = sdesc_at(opaque(d0), (uint32_t)(kQBytes + (c % kStages) * kHalfTile), 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + 256 + 128 * half, tS + kk * 8, sdesc_at(dv, kk * 2048, 16384), kIdescPV,
                    (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(b_empty + 8 * (c % kStages));
          ++c;
        }
        umma_commit(b_o);
        return true;
      };
      if (ok) ok = qk(0);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n && !(ok = qk(j + 1))) break;
        if (!mbar_wait(b_p, (uint32_t)j & 1u, ab, 134)) { ok = false; break; }
        tc_fence_after();
        ok = pv(j);
      }
      if (ok) umma_commit(b_of);  // every P.V done: O is final
      if (!ok) {  // let issued MMAs finish before tensor memory is released
        umma_commit(b_drain);
        mbar_wait_drain(b_drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int tid = threadIdx.x - 128;
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const uint32_t tO = tmem_addr(tmem, lane_base, 256);
    const int row = row0 + tid;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    float m_ref = kNegInf256, l_sum = 0.f, l_rnd = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!kFused && j == n - 1 && row < it.q1 && !(it.flags & kFirstStep)) {
        // last tile: bring this row's running (O, LSE) towards L2 for the merge
        const char* orow = reinterpret_cast<const char*>(p.o_run + ((size_t)row * p.Hq + h) * kD);
#pragma unroll
        for (int cb = 0; cb < kD * 4; cb += 128) prefetch_l2(orow + cb);
        prefetch_l2(p.lse + (size_t)h * p.T + row);
      }
      if (!mbar_wait(b_s + 8 * (j & 1), (uint32_t)(j >> 1) & 1u, ab, 135)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem_addr(tmem, lane_base, (uint32_t)(j & 1) * 128);
      uint32_t r[4][32];
      tmem_ld32(tS + 0, r[0]);
      tmem_ld32(tS + 32, r[1]);
      tmem_ld32(tS + 64, r[2]);
      tmem_ld32(tS + 96, r[3]);
      tmem_ld_wait();
      reg_fence32(r[0]); reg_fence32(r[1]); reg_fence32(r[2]); reg_fence32(r[3]);
      const int kst = tl.start(j), kend = tl.end(j);
      const bool need_mask = (kst + 128 > kend) || (p.causal && kst + 127 > row0);
      if (need_mask) {
        const int lim = p.causal ? min(kend - 1, row) : kend - 1;
#pragma unroll
        for (int cc = 0; cc < 128; ++cc)
          if (kst + cc > lim) r[cc >> 5][cc & 31] = __float_as_uint(kNegInf256);
      }
      uint64_t nm2 = 0, ls_a = 0, ls_b = 0;
      float lr0 = 0.f, lr1 = 0.f, lr2 = 0.f, lr3 = 0.f;
      auto p_chunk = [&](int cch) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t x =
              f2_fma(f2_pack(__uint_as_float(r[cch][2 * i]), __uint_as_float(r[cch][2 * i + 1])), sl2x2, nm2);
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
        tmem_st16(tS + 16 * cch, pk);
      };
      auto p_tile = [&](float m_use) {
        nm2 = f2_pack(-m_use, -m_use);
        ls_a = ls_b = 0;
        lr0 = lr1 = lr2 = lr3 = 0.f;
#pragma unroll
        for (int cch = 0; cch < 4; ++cch) p_chunk(cch);
      };
      auto tile_sum = [&]() {
        float a0, a1, b0, b1;
        f2_unpack(ls_a, a0, a1);
        f2_unpack(ls_b, b0, b1);
        return (a0 + a1) + (b0 + b1);
      };
      // speculate on the running reference maximum; take the row maximum (and
      // redo the tile) only when the tile's P would grow too large
      bool exact = __any_sync(0xffffffffu, m_ref == kNegInf256);
      bool rescale = false;
      float alpha = 1.f;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (exact) {
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = kNegInf256;
#pragma unroll
          for (int i = 0; i < 16; i += 2)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx[k] = fmax3(mx[k], __uint_as_float(r[k >> 1][16 * (k & 1) + i]),
                            __uint_as_float(r[k >> 1][16 * (k & 1) + i + 1]));
          const float m_tile =
              fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7]))) * sl2;
          const float m_new = fmaxf(m_ref, m_tile);
          rescale = m_new > m_ref + kRescaleThreshold256;
          if (rescale) {
            // integral reference (log2 units): partials over any split of the
            // keys differ by exact powers of two
            const float m_int = ceilf(m_new);
            alpha = ex2_approx(m_ref - m_int);
            l_sum *= alpha;
            l_rnd *= alpha;
            m_ref = m_int;
          }
        }
        p_tile((m_ref == kNegInf256) ? 0.f : m_ref);
        if (exact || !__any_sync(0xffffffffu, !(tile_sum() <= kSpecSumLimit256))) break;
        tmem_st_wait();  // the redo overwrites these P stores
        exact = true;
      }
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O holds P.V of tiles 0 .. j-1 once P(j-1).V(j-1) has completed.  S(j)
        // was committed after P(j-2).V(j-2) was issued and P(j).V(j) waits for
        // this warpgroup, so b_o has completed j-1 or j phases: a parity wait
        // on phase j-1 is exact.
        if (!mbar_wait(b_o, (uint32_t)(j - 1) & 1u, ab, 136)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int cch = 0; cch < kD / 32; ++cch) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * cch, o);
          tmem_ld_wait();
          reg_fence32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + 32 * cch, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p);
      l_sum += tile_sum();
      l_rnd += (lr0 + lr1) + (lr2 + lr3);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && (n > 0 || (it.flags & kFirstStep))) {
      if (n > 0) {
        ok = mbar_wait(b_of, 0, ab, 137);  // O final
        tc_fence_after();
      }
      ok = __all_sync(0xffffffffu, ok);
      // Rows leave through this warp's slice of the (now idle) Q buffer, four
      // passes of 64 columns, so every global load and store instruction
      // covers whole 256-byte row segments (two rows per instruction).
      constexpr int kW = 64;              // columns per pass
      constexpr int kChunks = kW / 4;     // 16-byte chunks of a row per pass
      constexpr int kPer = 32 / kChunks;  // rows per instruction
      constexpr int kSteps = 32 / kPer;   // instructions per pass
      const uint32_t scratch = sQ + (uint32_t)(warp & 3) * (kQBytes / 4);
      const int sub = lane / kChunks, ch = lane % kChunks;
      const int wrow0 = row0 + (int)lane_base;
      const size_t rstride = (size_t)p.Hq * kD;
      const bool valid = row < it.q1;
      const float lse_b = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) * kLn2_256 : kNegInf256;
      const float inv_l = (l_rnd > 0.f) ? 1.f / l_rnd : 0.f;
      auto stage_pass = [&](int ps, float w) {
#pragma unroll
        for (int cc = 0; cc < kW / 32; ++cc) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(tO + ps * kW + 32 * cc, o);
            tmem_ld_wait();
            reg_fence32(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int kc = 8 * cc + k;
            const uint32_t addr = scratch + (uint32_t)lane * (kW * 4) + (uint32_t)((kc ^ (lane % kChunks)) << 4);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                         "f"(__uint_as_float(o[4 * k]) * w), "f"(__uint_as_float(o[4 * k + 1]) * w),
                         "f"(__uint_as_float(o[4 * k + 2]) * w), "f"(__uint_as_float(o[4 * k + 3]) * w)
                         : "memory");
          }
        }
        __syncwarp();
      };
      auto read_staged = [&](int i) {
        const int rr = kPer * i + sub;
        float4 v;
        const uint32_t addr = scratch + (uint32_t)rr * (kW * 4) + (uint32_t)((ch ^ (rr % kChunks)) << 4);
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
        return v;
      };
      if (ok && kFused) {
        // the whole ring is done: O = (sum of P V) / (sum of the bf16 P), final LSE
        if (valid) p.lse[(size_t)h * p.T + row] = lse_b;
        const size_t obase = ((size_t)wrow0 * p.Hq + h) * kD + 4 * ch;
#pragma unroll 1
        for (int ps = 0; ps < kD / kW; ++ps) {
          stage_pass(ps, inv_l);
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int rr = kPer * i + sub;
            const float4 v = read_staged(i);
            if (wrow0 + rr >= it.q1) continue;
            const size_t off = obase + rr * rstride + ps * kW;
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
        const bool first = (it.flags & kFirstStep) != 0;
        float* lse_ptr = p.lse + (size_t)h * p.T + row;
        const float lse_a = (valid && !first) ? *lse_ptr : kNegInf256;
        float wa = 0.f, wb = 1.f, lse_new = lse_b;
        if (lse_b == kNegInf256) { wa = 1.f; wb = 0.f; lse_new = lse_a; }
        else if (lse_a != kNegInf256) {
          const float a2 = lse_a * 1.4426950408889634f, b2 = lse_b * 1.4426950408889634f;
          const float mx = fmaxf(a2, b2);
          const float n2 = mx + log2f(1.f + exp2f(-fabsf(a2 - b2)));
          wa = exp2f(a2 - n2);
          wb = exp2f(b2 - n2);
          lse_new = n2 * kLn2_256;
        }
        wb *= inv_l;
        const bool write = valid && (first || lse_b != kNegInf256);
        const bool read_old = valid && !first && lse_a != kNegInf256 && lse_b != kNegInf256;
        float* obase = p.o_run + ((size_t)wrow0 * p.Hq + h) * kD + 4 * ch;
#pragma unroll 1
        for (int ps = 0; ps < kD / kW; ++ps) {
          float4 old[kSteps];
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int rr = kPer * i + sub;
            const bool ro = __shfl_sync(0xffffffffu, read_old, rr) != 0;
            old[i] = ro ? *reinterpret_cast<const float4*>(obase + rr * rstride + ps * kW)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          stage_pass(ps, wb);
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int rr = kPer * i + sub;
            const float w = __shfl_sync(0xffffffffu, wa, rr);
            const bool ro = __shfl_sync(0xffffffffu, read_old, rr) != 0;
            const bool wr = __shfl_sync(0xffffffffu, write, rr) != 0;
            float4 v = read_staged(i);
            if (ro) {
              const float4 u = old[i];
              v.x = fmaf(w, u.x, v.x);
              v.y = fmaf(w, u.y, v.y);
              v.z = fmaf(w, u.z, v.z);
              v.w = fmaf(w, u.w, v.w);
            }
            if (wr) *reinterpret_cast<float4*>(obase + rr * rstride + ps * kW) = v;
          }
          __syncwarp();  // the next pass reuses the slice
        }
        if (write) *lse_ptr = lse_new;
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

template <bool kFused>
cudaError_t launch256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                      int num_items, cudaStream_t stream) {
  auto kern = ring_fwd_d256_kernel<kFused>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)num_items * p.Hq;
  if (grid <= 0) return cudaSuccess;
  FwdParams q = p;
  if (!kFused) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    q.next_cta = sms;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
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

cudaError_t launch_fwd_step_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const FwdParams& p, int num_items, cudaStream_t stream) {
  return launch256<false>(tq, tk, tv, p, num_items, stream);
}

cudaError_t launch_fwd_fused_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const FwdParams& p, int num_items, cudaStream_t stream) {
  return launch256<true>(tq, tk, tv, p, num_items, stream);
}

}  // namespace ra
