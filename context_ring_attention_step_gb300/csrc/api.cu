// api.cu -- the C ABI of ring_attn.h: host planner (sharding, ring pairing,
// work items), argument validation, TMA descriptor encoding and the per-step
// launch sequence.  The plan is host memory only; the device sees it through
// a copy into the caller's workspace at every call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/ring_attn.h"
#include "ring_attn_internal.h"

namespace ra {
// aux_kernels.cu: zero `header_bytes` at `header` and copy up to two work
// lists (device-visible pinned host memory -> workspace); byte counts are
// multiples of 16.
cudaError_t launch_ws_init(void* header, size_t header_bytes, const void* src0, void* dst0, size_t bytes0,
                          const void* src1, void* dst1, size_t bytes1, cudaStream_t stream);
}  // namespace ra

using ra::BwdItem;
using ra::FwdItem;

struct ra_plan {
  int32_t T = 0, num_docs = 0, Hq = 0, Hkv = 0, D = 0, causal = 1, layout = 1, steps = 0;
  int32_t bwd_cta_pairs = 0;  // head_dim 128 backward on CTA pairs (ra_plan_set_bwd_cta_pairs)
  float scale = 0.f;
  std::vector<int32_t> cu, cp;
  std::vector<FwdItem> fwd;
  std::vector<int64_t> fwd_off;  // steps + 1
  std::vector<BwdItem> bwd;
  std::vector<int64_t> bwd_off;  // steps + 1
  // The same items again, grouped by the query shard that computes them (the
  // rank of a multi-GPU ring: it keeps its query shard and sees key/value
  // shard (rank - s) mod cp at step s).  Items of (step s, rank r) are
  // [off[s * steps + r], off[s * steps + r + 1]).
  std::vector<FwdItem> fwd_rank;
  std::vector<int64_t> fwd_rank_off;
  std::vector<BwdItem> bwd_rank;
  std::vector<int64_t> bwd_rank_off;
  // single-launch forward over all ring steps: items (kb0 = first tile, ke0 =
  // tile count, kb1/ke1 = active tiles of the two 128-row query tiles) and the
  // key tiles, (start, range end) per tile, ring step by ring step
  std::vector<FwdItem> ffw;
  std::vector<int32_t> ftiles;
  int64_t visible_pairs = 0;
  // The work lists again, in device-visible pinned host memory (each list
  // padded to 16 bytes): a call's workspace set-up is then one small kernel
  // on its stream, not a copy-engine transfer from pageable memory (which can
  // block the host and queue behind the caller's own large copies).  Null
  // where pinned memory is unavailable; the calls then copy from the vectors.
  uint8_t* staged = nullptr;
  const uint8_t* staged_dev = nullptr;
  size_t st_fwd = 0, st_bwd = 0, st_ffw = 0, st_tiles = 0, st_fwdr = 0, st_bwdr = 0;
  ~ra_plan() {
    if (staged) cudaFreeHost(staged);
  }
};

namespace {

thread_local std::string g_err;

ra_status fail(ra_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

constexpr size_t kHeader = 256;
constexpr int kSelfTestSite = 900;  // status code of the failure-detection self-test
constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Chunk boundaries of one document of length L (document-local):
// zigzag -> 2*cp chunks, contiguous -> cp chunks, floor(k L / n).
int32_t bound(int32_t L, int32_t n, int32_t k) { return (int32_t)(((int64_t)k * L) / n); }

// Shard r of a document: up to two local ranges (zigzag: chunk r, chunk 2cp-1-r).
int shard(int32_t L, int32_t cp, int32_t layout, int32_t r, int32_t* b, int32_t* e) {
  if (layout == RA_LAYOUT_ZIGZAG) {
    const int32_t n = 2 * cp;
    b[0] = bound(L, n, r);
    e[0] = bound(L, n, r + 1);
    b[1] = bound(L, n, n - 1 - r);
    e[1] = bound(L, n, n - r);
    return 2;
  }
  b[0] = bound(L, cp, r);
  e[0] = bound(L, cp, r + 1);
  return 1;
}

int32_t tiles128(int32_t a, int32_t b) { return b > a ? (b - a + 127) / 128 : 0; }

// The backward on CTA pairs over two key tiles (head_dim 128, when asked for).
bool bwd_pairs(const ra_plan& P) { return P.D == 128 && P.bwd_cta_pairs != 0; }

// Query rows of one forward CTA: two 128-row tiles at head_dim 64/128, one at
// head_dim 256 (whose output accumulator alone takes half of tensor memory).
int32_t rows_per_item(const ra_plan& P) { return P.D == 256 ? 128 : 256; }

void build_items(ra_plan& P) {
  P.fwd.clear();
  P.bwd.clear();
  P.fwd_off.assign(1, 0);
  P.bwd_off.assign(1, 0);
  P.fwd_rank.clear();
  P.bwd_rank.clear();
  P.fwd_rank_off.assign(1, 0);
  P.bwd_rank_off.assign(1, 0);
  auto by_tiles = [](const auto& a, const auto& b) { return a.tiles > b.tiles; };
  for (int32_t s = 0; s < P.steps; ++s) {
    std::vector<FwdItem> fs;
    std::vector<BwdItem> bs;
    std::vector<std::vector<FwdItem>> fr(P.steps);  // by query shard
    std::vector<std::vector<BwdItem>> br(P.steps);
    for (int32_t d = 0; d < P.num_docs; ++d) {
      const int32_t base = P.cu[d], L = P.cu[d + 1] - P.cu[d], cp = P.cp[d];
      if (L == 0 || s >= cp) continue;
      for (int32_t r = 0; r < cp; ++r) {
        // ---- forward: query shard r meets key/value shard j = (r - s) mod cp
        const int32_t j = ((r - s) % cp + cp) % cp;
        int32_t qb[2], qe[2], kb[2], ke[2];
        const int nq = shard(L, cp, P.layout, r, qb, qe);
        const int nk = shard(L, cp, P.layout, j, kb, ke);
        for (int a = 0; a < nq; ++a) {
          for (int32_t q0 = base + qb[a]; q0 < base + qe[a]; q0 += rows_per_item(P)) {
            const int32_t q1 = std::min(q0 + rows_per_item(P), base + qe[a]);
            FwdItem it{};
            it.q0 = q0;
            it.q1 = q1;
            int32_t rb[2] = {0, 0}, re[2] = {0, 0};
            int nr = 0;
            for (int c = 0; c < nk; ++c) {
              int32_t b = base + kb[c], e = base + ke[c];
              if (P.causal) e = std::min(e, q1);
              if (e > b) { rb[nr] = b; re[nr] = e; ++nr; }
            }
            if (nr == 0) continue;
            it.kb0 = rb[0]; it.ke0 = re[0];
            it.kb1 = nr > 1 ? rb[1] : 0; it.ke1 = nr > 1 ? re[1] : 0;
            it.flags = s == 0 ? ra::kFirstStep : 0;
            it.tiles = tiles128(it.kb0, it.ke0) + tiles128(it.kb1, it.ke1);
            fs.push_back(it);
            fr[r].push_back(it);
          }
        }
        // ---- backward: key/value shard r is held by query shard (r + s) mod cp.
        // One item per (key tile, key/value head), grouped by shard pair and
        // head: the CTAs running together then reduce into the dQ rows of one
        // query shard and one GQA group, a working set that stays in L2.  At
        // head_dim 128 the items come in pairs, neighbouring key tiles of one
        // range for the two CTAs of a cluster (bwd_pair.cu): both walk the query
        // rows the first tile meets (a superset of the second's; the rest is
        // masked), and a range with an odd number of tiles ends in an empty one.
        const int32_t qr = (r + s) % cp;
        int32_t kb2[2], ke2[2], qb2[2], qe2[2];
        const int nk2 = shard(L, cp, P.layout, r, kb2, ke2);
        const int nq2 = shard(L, cp, P.layout, qr, qb2, qe2);
        const bool pairs = bwd_pairs(P);
        for (int32_t g = 0; g < P.Hkv; ++g)
        for (int a = 0; a < nk2; ++a) {
          const int32_t ke = base + ke2[a];
          for (int32_t k0 = base + kb2[a]; k0 < ke; k0 += pairs ? 256 : 128) {
            const int32_t k1 = std::min(k0 + 128, ke);
            BwdItem it{};
            it.k0 = k0;
            it.k1 = k1;
            int32_t rb[2] = {0, 0}, re[2] = {0, 0};
            int nr = 0;
            for (int c = 0; c < nq2; ++c) {
              int32_t b = base + qb2[c], e = base + qe2[c];
              if (P.causal) b = std::max(b, k0);
              if (e > b) { rb[nr] = b; re[nr] = e; ++nr; }
            }
            if (nr == 0) continue;
            it.qb0 = rb[0]; it.qe0 = re[0];
            it.qb1 = nr > 1 ? rb[1] : 0; it.qe1 = nr > 1 ? re[1] : 0;
            it.flags = (s == 0 ? ra::kFirstStep : 0) | (g << ra::kHeadShift);
            it.tiles = tiles128(it.qb0, it.qe0) + tiles128(it.qb1, it.qe1);
            bs.push_back(it);
            br[qr].push_back(it);
            if (pairs) {
              it.k0 = k1;
              it.k1 = std::min(k0 + 256, ke);
              bs.push_back(it);
              br[qr].push_back(it);
            }
          }
        }
      }
    }
    // forward: longest items first, so the tail of each step launch is short
    std::stable_sort(fs.begin(), fs.end(), by_tiles);
    P.fwd.insert(P.fwd.end(), fs.begin(), fs.end());
    P.bwd.insert(P.bwd.end(), bs.begin(), bs.end());
    P.fwd_off.push_back((int64_t)P.fwd.size());
    P.bwd_off.push_back((int64_t)P.bwd.size());
    for (int32_t r = 0; r < P.steps; ++r) {
      std::stable_sort(fr[r].begin(), fr[r].end(), by_tiles);
      P.fwd_rank.insert(P.fwd_rank.end(), fr[r].begin(), fr[r].end());
      P.bwd_rank.insert(P.bwd_rank.end(), br[r].begin(), br[r].end());
      P.fwd_rank_off.push_back((int64_t)P.fwd_rank.size());
      P.bwd_rank_off.push_back((int64_t)P.bwd_rank.size());
    }
  }
}

// Work list of the single-launch forward: one item per 256-row query chunk,
// holding every key tile the chunk meets over the whole ring, in ring order
// (step s: the key/value shard (r - s) mod cp, its ranges in ascending order),
// causally clipped to keys < q1.  The running (O, LSE) of the chunk then stays
// on chip from the first ring step to the last: each step's partial is merged
// by continuing the online softmax instead of through HBM.
void build_fused(ra_plan& P) {
  P.ffw.clear();
  P.ftiles.clear();
  for (int32_t d = 0; d < P.num_docs; ++d) {
    const int32_t base = P.cu[d], L = P.cu[d + 1] - P.cu[d], cp = P.cp[d];
    if (L == 0) continue;
    for (int32_t r = 0; r < cp; ++r) {
      int32_t qb[2], qe[2];
      const int nq = shard(L, cp, P.layout, r, qb, qe);
      for (int a = 0; a < nq; ++a) {
        for (int32_t q0 = base + qb[a]; q0 < base + qe[a]; q0 += rows_per_item(P)) {
          const int32_t q1 = std::min(q0 + rows_per_item(P), base + qe[a]);
          const int32_t last0 = std::min(q0 + 128, q1) - 1, last1 = q1 - 1;
          const bool two = q0 + 128 < q1;
          FwdItem it{};
          it.q0 = q0;
          it.q1 = q1;
          it.kb0 = (int32_t)(P.ftiles.size() / 2);
          int32_t n = 0, na0 = 0, na1 = 0;
          for (int32_t s = 0; s < cp; ++s) {
            const int32_t j = ((r - s) % cp + cp) % cp;
            int32_t kb[2], ke[2];
            const int nk = shard(L, cp, P.layout, j, kb, ke);
            for (int c = 0; c < nk; ++c) {
              const int32_t b = base + kb[c];
              const int32_t e = P.causal ? std::min(base + ke[c], q1) : base + ke[c];
              for (int32_t kst = b; kst < e; kst += 128) {
                P.ftiles.push_back(kst);
                P.ftiles.push_back(e);
                ++n;
                if (!P.causal || kst <= last0) ++na0;
                if (two && (!P.causal || kst <= last1)) ++na1;
              }
            }
          }
          if (n == 0) continue;
          it.ke0 = n;
          it.kb1 = na0;
          it.ke1 = na1;
          it.flags = ra::kFirstStep;
          it.tiles = n;
          P.ffw.push_back(it);
        }
      }
    }
  }
  // longest first: the grid's tail is short
  std::stable_sort(P.ffw.begin(), P.ffw.end(), [](const FwdItem& a, const FwdItem& b) { return a.tiles > b.tiles; });
}

// Row pitch (in floats) of the backward's per-head Delta and LSE*log2(e)
// rows: T rounded up to 4, so every row starts 16-byte aligned for TMA.
int64_t stat_pitch(const ra_plan& P) { return ((int64_t)P.T + 3) & ~int64_t(3); }

struct FwdLayout {
  size_t items, ritems, orun, total;
};
struct FusedLayout {
  size_t items, tiles, total;
};
struct BwdLayout {
  size_t items, ritems, delta, lse2, dq, dk, dv, total;
};

FwdLayout fwd_layout(const ra_plan& P, int o_fp32) {
  FwdLayout l{};
  size_t off = kHeader;
  l.items = off;
  off = align256(off + P.fwd.size() * sizeof(FwdItem));
  l.ritems = off;
  off = align256(off + P.fwd_rank.size() * sizeof(FwdItem));
  l.orun = off;
  if (!o_fp32) off = align256(off + (size_t)P.T * P.Hq * P.D * 4);
  l.total = off;
  return l;
}

FusedLayout fused_layout(const ra_plan& P) {
  FusedLayout l{};
  size_t off = kHeader;
  l.items = off;
  off = align256(off + P.ffw.size() * sizeof(FwdItem));
  l.tiles = off;
  off = align256(off + P.ftiles.size() * sizeof(int32_t));
  l.total = off;
  return l;
}

BwdLayout bwd_layout(const ra_plan& P, int g_fp32) {
  BwdLayout l{};
  size_t off = kHeader;
  l.items = off;
  off = align256(off + P.bwd.size() * sizeof(BwdItem));
  l.ritems = off;
  off = align256(off + P.bwd_rank.size() * sizeof(BwdItem));
  l.delta = off;
  off = align256(off + (size_t)P.Hq * stat_pitch(P) * 4);
  l.lse2 = off;
  off = align256(off + (size_t)P.Hq * stat_pitch(P) * 4);
  l.dq = l.dk = l.dv = 0;
  if (!g_fp32) {
    l.dq = off;
    off = align256(off + (size_t)P.T * P.Hq * P.D * 4);
    l.dk = off;
    off = align256(off + (size_t)P.T * P.Hkv * P.D * 4);
    l.dv = off;
    off = align256(off + (size_t)P.T * P.Hkv * P.D * 4);
  }
  l.total = off;
  return l;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// THD bf16 tensor [T, H, D] as a 3-D map {D, H, T}; box {64, 1, rows} (rows = 128,
// or 64 for the head_dim 256 backward's query tiles), 128-byte swizzle.
bool encode_thd(CUtensorMap* m, const void* base, int T, int H, int D, int rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-head fp32 rows [Hq, pitch] as a 2-D map {pitch, Hq}; box {width, 1}.
bool encode_rows(CUtensorMap* m, const void* base, int64_t pitch, int H, int width = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)pitch, (cuuint64_t)H};
  cuuint64_t strides[1] = {(cuuint64_t)pitch * 4};
  cuuint32_t box[2] = {(cuuint32_t)width, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 THD accumulator [T, H, D] as a 3-D map {D, H, T}; box {32, 1, 32}
// (128 bytes x 32 rows, one warp's rows), 128-byte swizzle: the target of the
// dQ reductions.
bool encode_acc(CUtensorMap* m, const void* base, int T, int H, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  cuuint32_t box[3] = {32, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t pad16(size_t b) { return (b + 15) & ~size_t(15); }

// Copy the work lists into mapped pinned host memory (see ra_plan::staged).
void stage_work_lists(ra_plan& P) {
  const size_t bf = pad16(P.fwd.size() * sizeof(FwdItem)), bb = pad16(P.bwd.size() * sizeof(BwdItem));
  const size_t bu = pad16(P.ffw.size() * sizeof(FwdItem)), bt = pad16(P.ftiles.size() * sizeof(int32_t));
  const size_t bfr = pad16(P.fwd_rank.size() * sizeof(FwdItem)), bbr = pad16(P.bwd_rank.size() * sizeof(BwdItem));
  const size_t total = bf + bb + bu + bt + bfr + bbr;
  if (total == 0) return;
  const char* off = std::getenv("RA_NO_PINNED_WORK_LISTS");  // tests of the copy fallback
  if (off && off[0] == '1') return;
  void* h = nullptr;
  if (cudaHostAlloc(&h, total, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    (void)cudaGetLastError();  // no usable device here: the calls copy from the vectors
    return;
  }
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    cudaFreeHost(h);
    return;
  }
  uint8_t* b = static_cast<uint8_t*>(h);
  std::memset(b, 0, total);
  P.st_fwd = 0;
  P.st_bwd = bf;
  P.st_ffw = bf + bb;
  P.st_tiles = bf + bb + bu;
  P.st_fwdr = bf + bb + bu + bt;
  P.st_bwdr = bf + bb + bu + bt + bfr;
  if (!P.fwd.empty()) std::memcpy(b + P.st_fwd, P.fwd.data(), P.fwd.size() * sizeof(FwdItem));
  if (!P.bwd.empty()) std::memcpy(b + P.st_bwd, P.bwd.data(), P.bwd.size() * sizeof(BwdItem));
  if (!P.ffw.empty()) std::memcpy(b + P.st_ffw, P.ffw.data(), P.ffw.size() * sizeof(FwdItem));
  if (!P.ftiles.empty()) std::memcpy(b + P.st_tiles, P.ftiles.data(), P.ftiles.size() * sizeof(int32_t));
  if (!P.fwd_rank.empty()) std::memcpy(b + P.st_fwdr, P.fwd_rank.data(), P.fwd_rank.size() * sizeof(FwdItem));
  if (!P.bwd_rank.empty()) std::memcpy(b + P.st_bwdr, P.bwd_rank.data(), P.bwd_rank.size() * sizeof(BwdItem));
  P.staged = b;
  P.staged_dev = static_cast<const uint8_t*>(d);
}

// Zero the workspace's status header and put up to two work lists in place:
// (staged offset, host copy, bytes, workspace offset) per list.
cudaError_t ws_setup(const ra_plan* P, uint8_t* ws, cudaStream_t st, size_t so0, const void* h0, size_t b0,
                     size_t d0, size_t so1 = 0, const void* h1 = nullptr, size_t b1 = 0, size_t d1 = 0) {
  if (P->staged_dev)
    return ra::launch_ws_init(ws, kHeader, P->staged_dev + so0, ws + d0, b0 ? pad16(b0) : 0, P->staged_dev + so1,
                              ws + d1, b1 ? pad16(b1) : 0, st);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e == cudaSuccess && b0) e = cudaMemcpyAsync(ws + d0, h0, b0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && b1) e = cudaMemcpyAsync(ws + d1, h1, b1, cudaMemcpyHostToDevice, st);
  return e;
}

ra_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

namespace ra {
ra_status set_last_error(ra_status st, const char* msg) {
  g_err = msg;
  return st;
}
}  // namespace ra

extern "C" {

int32_t ra_abi_version(void) { return 2; }

const char* ra_last_error(void) { return g_err.c_str(); }

ra_status ra_plan_create(ra_plan** out, const int32_t* cu_seqlens, int32_t num_docs, const int32_t* cp_size_per_doc,
                         int32_t cp_size, int32_t layout, int32_t causal, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, float softmax_scale) {
  if (!out) return fail(RA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cu_seqlens) return fail(RA_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (num_docs < 1) return fail(RA_ERR_INVALID_ARG, "num_docs must be >= 1 (got %d)", num_docs);
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG)
    return fail(RA_ERR_INVALID_ARG, "layout must be 0 (contiguous) or 1 (zigzag), got %d", layout);
  if (causal != 0 && causal != 1) return fail(RA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return fail(RA_ERR_INVALID_ARG, "need Hq >= 1, Hkv >= 1 and Hq %% Hkv == 0 (got %d, %d)", num_q_heads,
                num_kv_heads);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(RA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale))
    return fail(RA_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (cu_seqlens[0] != 0) return fail(RA_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
  for (int32_t d = 0; d < num_docs; ++d)
    if (cu_seqlens[d + 1] < cu_seqlens[d])
      return fail(RA_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing (index %d)", d + 1);
  const int64_t T = cu_seqlens[num_docs];
  if (T < 1) return fail(RA_ERR_INVALID_ARG, "total tokens must be >= 1");
  if (T * (int64_t)std::max(num_q_heads, num_kv_heads) * head_dim >= ((int64_t)1 << 40))
    return fail(RA_ERR_UNSUPPORTED, "problem too large");
  ra_plan* P = new (std::nothrow) ra_plan();
  if (!P) return fail(RA_ERR_INVALID_ARG, "out of host memory");
  P->T = (int32_t)T;
  P->num_docs = num_docs;
  P->Hq = num_q_heads;
  P->Hkv = num_kv_heads;
  P->D = head_dim;
  P->causal = causal;
  P->layout = layout;
  P->scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)head_dim);
  P->cu.assign(cu_seqlens, cu_seqlens + num_docs + 1);
  P->cp.resize(num_docs);
  for (int32_t d = 0; d < num_docs; ++d) {
    const int32_t c = cp_size_per_doc ? cp_size_per_doc[d] : cp_size;
    if (c < 1 || c > 4096) {
      delete P;
      return fail(RA_ERR_INVALID_ARG, "cp_size of document %d must be in [1, 4096] (got %d)", d, c);
    }
    P->cp[d] = c;
    P->steps = std::max(P->steps, c);
    const int64_t L = cu_seqlens[d + 1] - cu_seqlens[d];
    P->visible_pairs += causal ? L * (L + 1) / 2 : L * L;
  }
  build_items(*P);
  build_fused(*P);
  stage_work_lists(*P);
  *out = P;
  return RA_OK;
}

void ra_plan_destroy(ra_plan* plan) { delete plan; }

ra_status ra_plan_set_bwd_cta_pairs(ra_plan* P, int32_t on) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (on != 0 && on != 1) return fail(RA_ERR_INVALID_ARG, "on must be 0 or 1 (got %d)", on);
  if (on && P->D != 128) return fail(RA_ERR_UNSUPPORTED, "the CTA-pair backward needs head_dim 128 (got %d)", P->D);
  if (P->bwd_cta_pairs == on) return RA_OK;
  P->bwd_cta_pairs = on;
  build_items(*P);  // the backward items pair up (or not); the forward lists are rebuilt unchanged
  if (P->staged) {
    cudaFreeHost(P->staged);
    P->staged = nullptr;
    P->staged_dev = nullptr;
  }
  stage_work_lists(*P);
  return RA_OK;
}

ra_status ra_plan_workspace_bytes(const ra_plan* P, int32_t o_is_fp32, int32_t grads_fp32, size_t* fwd_bytes,
                                  size_t* bwd_bytes) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  (void)o_is_fp32;  // ra_fwd writes its output once, in its final dtype: no running output
  if (fwd_bytes) *fwd_bytes = fused_layout(*P).total;
  if (bwd_bytes) *bwd_bytes = bwd_layout(*P, grads_fp32).total;
  return RA_OK;
}

ra_status ra_plan_ring_step_workspace_bytes(const ra_plan* P, int32_t o_is_fp32, size_t* fwd_bytes) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!fwd_bytes) return fail(RA_ERR_INVALID_ARG, "fwd_bytes is NULL");
  *fwd_bytes = fwd_layout(*P, o_is_fp32).total;
  return RA_OK;
}

ra_status ra_plan_stats(const ra_plan* P, int32_t* num_steps, int64_t* visible_pairs, int64_t* fwd_items,
                        int64_t* bwd_items) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (num_steps) *num_steps = P->steps;
  if (visible_pairs) *visible_pairs = P->visible_pairs;
  if (fwd_items) *fwd_items = (int64_t)P->fwd.size();
  if (bwd_items) *bwd_items = (int64_t)P->bwd.size();
  return RA_OK;
}

ra_status ra_plan_work_items(const ra_plan* P, int32_t which, int32_t* items, int64_t capacity,
                             int64_t* step_offsets, int64_t* count) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (which != 0 && which != 1) return fail(RA_ERR_INVALID_ARG, "which must be 0 (fwd) or 1 (bwd)");
  static_assert(sizeof(FwdItem) == 32 && sizeof(BwdItem) == 32, "work items are 8 x int32");
  const size_t n = which == 0 ? P->fwd.size() : P->bwd.size();
  if (count) *count = (int64_t)n;
  if (items) {
    if (capacity < (int64_t)n) return fail(RA_ERR_INVALID_ARG, "capacity %lld < %zu items", (long long)capacity, n);
    if (n) std::memcpy(items, which == 0 ? (const void*)P->fwd.data() : (const void*)P->bwd.data(), n * 32);
  }
  if (step_offsets) {
    const std::vector<int64_t>& off = which == 0 ? P->fwd_off : P->bwd_off;
    std::copy(off.begin(), off.end(), step_offsets);
  }
  return RA_OK;
}

ra_status ra_plan_rank_work_items(const ra_plan* P, int32_t which, int32_t* items, int64_t capacity,
                                  int64_t* offsets, int64_t* count) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (which != 0 && which != 1) return fail(RA_ERR_INVALID_ARG, "which must be 0 (fwd) or 1 (bwd)");
  const size_t n = which == 0 ? P->fwd_rank.size() : P->bwd_rank.size();
  if (count) *count = (int64_t)n;
  if (items) {
    if (capacity < (int64_t)n) return fail(RA_ERR_INVALID_ARG, "capacity %lld < %zu items", (long long)capacity, n);
    if (n) std::memcpy(items, which == 0 ? (const void*)P->fwd_rank.data() : (const void*)P->bwd_rank.data(), n * 32);
  }
  if (offsets) {
    const std::vector<int64_t>& off = which == 0 ? P->fwd_rank_off : P->bwd_rank_off;
    std::copy(off.begin(), off.end(), offsets);
  }
  return RA_OK;
}

ra_status ra_shard_token_ranges(const ra_plan* P, int32_t doc, int32_t rank, int32_t* begin2, int32_t* end2,
                                int32_t* count) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!begin2 || !end2 || !count) return fail(RA_ERR_INVALID_ARG, "output pointer is NULL");
  if (doc < 0 || doc >= P->num_docs) return fail(RA_ERR_INVALID_ARG, "doc %d out of range", doc);
  if (rank < 0 || rank >= P->cp[doc]) return fail(RA_ERR_INVALID_ARG, "rank %d out of range", rank);
  const int32_t L = P->cu[doc + 1] - P->cu[doc];
  int32_t b[2], e[2];
  const int n = shard(L, P->cp[doc], P->layout, rank, b, e);
  for (int i = 0; i < n; ++i) {
    begin2[i] = P->cu[doc] + b[i];
    end2[i] = P->cu[doc] + e[i];
  }
  *count = n;
  return RA_OK;
}

// ---------------------------------------------------------------- forward

static ra_status check_fwd_ws(const ra_plan* P, int32_t o_is_fp32, const void* workspace, size_t bytes,
                              FwdLayout* L) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned16(workspace)) return fail(RA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  *L = fwd_layout(*P, o_is_fp32);
  if (bytes < L->total)
    return fail(RA_ERR_WORKSPACE, "workspace too small for the ring-step forward: %zu < %zu bytes "
                "(ra_plan_ring_step_workspace_bytes)", bytes, L->total);
  return RA_OK;
}

ra_status ra_fwd_prepare(const ra_plan* P, int32_t o_is_fp32, void* workspace, size_t workspace_bytes,
                         void* stream_) {
  FwdLayout L;
  ra_status rs = check_fwd_ws(P, o_is_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaError_t e = ws_setup(P, ws, st, P->st_fwd, P->fwd.data(), P->fwd.size() * sizeof(FwdItem), L.items,
                           P->st_fwdr, P->fwd_rank.data(), P->fwd_rank.size() * sizeof(FwdItem), L.ritems);
  if (e != cudaSuccess) return cuda_fail(e, "workspace set-up");
  return RA_OK;
}

// One forward ring-step launch over work items [first, first + n) of the list
// at workspace offset `list` (the per-step list or the per-rank one).
static ra_status fwd_step_launch(const ra_plan* P, size_t list, int64_t first, int64_t n, const void* q, const void* k,
                                 const void* v, void* o, int32_t o_is_fp32, float* lse, void* workspace,
                                 const FwdLayout& L, void* stream_) {
  if (!q || !k || !v || !o || !lse) return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(RA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (n == 0) return RA_OK;
  CUtensorMap tq, tk, tv;
  if (!encode_thd(&tq, q, P->T, P->Hq, P->D) || !encode_thd(&tk, k, P->T, P->Hkv, P->D) ||
      !encode_thd(&tv, v, P->T, P->Hkv, P->D))
    return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor)");
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  ra::FwdParams p{};
  p.items = reinterpret_cast<const FwdItem*>(ws + list) + first;
  p.Hq = P->Hq;
  p.Hkv = P->Hkv;
  p.T = P->T;
  p.causal = P->causal;
  p.scale_log2 = P->scale * 1.4426950408889634f;
  p.o_run = o_is_fp32 ? reinterpret_cast<float*>(o) : reinterpret_cast<float*>(ws + L.orun);
  p.lse = lse;
  p.status = reinterpret_cast<int*>(ws);
  cudaError_t e = ra::launch_fwd_step(P->D, tq, tk, tv, p, (int)n, reinterpret_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return cuda_fail(e, "forward step launch");
  return RA_OK;
}

ra_status ra_fwd_ring_step(const ra_plan* P, int32_t step, const void* q, const void* k, const void* v, void* o,
                           int32_t o_is_fp32, float* lse, void* workspace, size_t workspace_bytes, void* stream_) {
  FwdLayout L;
  ra_status rs = check_fwd_ws(P, o_is_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (step < 0 || step >= P->steps) return fail(RA_ERR_INVALID_ARG, "step %d outside [0, %d)", step, P->steps);
  return fwd_step_launch(P, L.items, P->fwd_off[step], P->fwd_off[step + 1] - P->fwd_off[step], q, k, v, o,
                         o_is_fp32, lse, workspace, L, stream_);
}

ra_status ra_fwd_ring_step_rank(const ra_plan* P, int32_t step, int32_t rank, const void* q, const void* k,
                                const void* v, void* o, int32_t o_is_fp32, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream_) {
  FwdLayout L;
  ra_status rs = check_fwd_ws(P, o_is_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (step < 0 || step >= P->steps) return fail(RA_ERR_INVALID_ARG, "step %d outside [0, %d)", step, P->steps);
  if (rank < 0 || rank >= P->steps) return fail(RA_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, P->steps);
  const int64_t c = (int64_t)step * P->steps + rank;
  return fwd_step_launch(P, L.ritems, P->fwd_rank_off[c], P->fwd_rank_off[c + 1] - P->fwd_rank_off[c], q, k, v, o,
                         o_is_fp32, lse, workspace, L, stream_);
}

ra_status ra_fwd_finish(const ra_plan* P, void* o, int32_t o_is_fp32, void* workspace, size_t workspace_bytes,
                        void* stream_) {
  FwdLayout L;
  ra_status rs = check_fwd_ws(P, o_is_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (!o || !aligned16(o)) return fail(RA_ERR_INVALID_ARG, "o must be a 16-byte aligned device pointer");
  if (o_is_fp32) return RA_OK;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaError_t e = ra::launch_cast_bf16(reinterpret_cast<const float*>(ws + L.orun), o, (size_t)P->T * P->Hq * P->D,
                                       reinterpret_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return cuda_fail(e, "output cast launch");
  return RA_OK;
}

ra_status ra_fwd_ring_steps(const ra_plan* P, const void* q, const void* k, const void* v, void* o,
                            int32_t o_is_fp32, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!q || !k || !v || !o || !lse || !workspace) return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
    return fail(RA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  ra_status rs = ra_fwd_prepare(P, o_is_fp32, workspace, workspace_bytes, stream);
  for (int32_t s = 0; s < P->steps && rs == RA_OK; ++s)
    rs = ra_fwd_ring_step(P, s, q, k, v, o, o_is_fp32, lse, workspace, workspace_bytes, stream);
  if (rs == RA_OK) rs = ra_fwd_finish(P, o, o_is_fp32, workspace, workspace_bytes, stream);
  return rs;
}

// ---------------------------------------------------------------- forward, one launch

ra_status ra_plan_fused_workspace_bytes(const ra_plan* P, size_t* fwd_bytes) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!fwd_bytes) return fail(RA_ERR_INVALID_ARG, "fwd_bytes is NULL");
  *fwd_bytes = fused_layout(*P).total;
  return RA_OK;
}

ra_status ra_plan_fused_items(const ra_plan* P, int32_t* items, int64_t item_capacity, int32_t* tiles,
                              int64_t tile_capacity, int64_t* num_items, int64_t* num_tiles) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  const int64_t ni = (int64_t)P->ffw.size(), nt = (int64_t)P->ftiles.size() / 2;
  if (num_items) *num_items = ni;
  if (num_tiles) *num_tiles = nt;
  if (items) {
    if (item_capacity < ni) return fail(RA_ERR_INVALID_ARG, "item capacity %lld < %lld", (long long)item_capacity, (long long)ni);
    if (ni) std::memcpy(items, P->ffw.data(), (size_t)ni * sizeof(FwdItem));
  }
  if (tiles) {
    if (tile_capacity < nt) return fail(RA_ERR_INVALID_ARG, "tile capacity %lld < %lld", (long long)tile_capacity, (long long)nt);
    if (nt) std::memcpy(tiles, P->ftiles.data(), (size_t)nt * 2 * sizeof(int32_t));
  }
  return RA_OK;
}

ra_status ra_fwd(const ra_plan* P, const void* q, const void* k, const void* v, void* o, int32_t o_is_fp32,
                 float* lse, void* workspace, size_t workspace_bytes, void* stream_) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!q || !k || !v || !o || !lse || !workspace) return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
    return fail(RA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  const FusedLayout L = fused_layout(*P);
  if (workspace_bytes < L.total)
    return fail(RA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", workspace_bytes, L.total);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaError_t e = ws_setup(P, ws, st, P->st_ffw, P->ffw.data(), P->ffw.size() * sizeof(FwdItem), L.items,
                           P->st_tiles, P->ftiles.data(), P->ftiles.size() * sizeof(int32_t), L.tiles);
  if (e != cudaSuccess) return cuda_fail(e, "workspace set-up");
  if (P->ffw.empty()) return RA_OK;
  CUtensorMap tq, tk, tv;
  if (!encode_thd(&tq, q, P->T, P->Hq, P->D) || !encode_thd(&tk, k, P->T, P->Hkv, P->D) ||
      !encode_thd(&tv, v, P->T, P->Hkv, P->D))
    return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor)");
  ra::FwdParams p{};
  p.items = reinterpret_cast<const FwdItem*>(ws + L.items);
  p.tiles = reinterpret_cast<const int2*>(ws + L.tiles);
  p.Hq = P->Hq;
  p.Hkv = P->Hkv;
  p.T = P->T;
  p.causal = P->causal;
  p.scale_log2 = P->scale * 1.4426950408889634f;
  p.o_out = o;
  p.o_bf16 = o_is_fp32 ? 0 : 1;
  p.lse = lse;
  p.status = reinterpret_cast<int*>(ws);
  e = ra::launch_fwd_fused(P->D, tq, tk, tv, p, (int)P->ffw.size(), st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return RA_OK;
}

ra_status ra_fwd_fused(const ra_plan* P, const void* q, const void* k, const void* v, void* o, int32_t o_is_fp32,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return ra_fwd(P, q, k, v, o, o_is_fp32, lse, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- backward

static ra_status check_bwd_ws(const ra_plan* P, int32_t grads_fp32, const void* workspace, size_t bytes,
                              BwdLayout* L) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned16(workspace)) return fail(RA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  *L = bwd_layout(*P, grads_fp32);
  if (bytes < L->total) return fail(RA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", bytes, L->total);
  return RA_OK;
}

static ra::BwdParams bwd_params(const ra_plan* P, const BwdLayout& L, uint8_t* ws, void* dq, void* dk, void* dv,
                                int32_t grads_fp32) {
  ra::BwdParams p{};
  p.Hq = P->Hq;
  p.Hkv = P->Hkv;
  p.T = P->T;
  p.causal = P->causal;
  p.scale = P->scale;
  p.scale_log2 = P->scale * 1.4426950408889634f;
  p.delta = reinterpret_cast<float*>(ws + L.delta);
  p.lse2 = reinterpret_cast<float*>(ws + L.lse2);
  p.stat_pitch = stat_pitch(*P);
  p.dq_acc = grads_fp32 ? reinterpret_cast<float*>(dq) : reinterpret_cast<float*>(ws + L.dq);
  p.dk_acc = grads_fp32 ? reinterpret_cast<float*>(dk) : reinterpret_cast<float*>(ws + L.dk);
  p.dv_acc = grads_fp32 ? reinterpret_cast<float*>(dv) : reinterpret_cast<float*>(ws + L.dv);
  p.status = reinterpret_cast<int*>(ws);
  return p;
}

ra_status ra_bwd_prepare(const ra_plan* P, const void* o, int32_t o_is_fp32, const void* dout, const float* lse,
                         void* dq, void* dk, void* dv, int32_t grads_fp32, void* workspace, size_t workspace_bytes,
                         void* stream_) {
  BwdLayout L;
  ra_status rs = check_bwd_ws(P, grads_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (!o || !dout || !lse || (grads_fp32 && (!dq || !dk || !dv)))
    return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      (grads_fp32 && (!aligned16(dq) || !aligned16(dk) || !aligned16(dv))))
    return fail(RA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaError_t e = ws_setup(P, ws, st, P->st_bwd, P->bwd.data(), P->bwd.size() * sizeof(BwdItem), L.items,
                           P->st_bwdr, P->bwd_rank.data(), P->bwd_rank.size() * sizeof(BwdItem), L.ritems);
  if (e != cudaSuccess) return cuda_fail(e, "workspace set-up");
  ra::BwdParams p = bwd_params(P, L, ws, dq, dk, dv, grads_fp32);
  // the row padding past T is read by the tile loads (and masked): keep it finite
  e = cudaMemsetAsync(ws + L.delta, 0, L.dq ? L.dq - L.delta : L.total - L.delta, st);
  if (e != cudaSuccess) return cuda_fail(e, "stat reset");
  e = ra::launch_bwd_preprocess(o, o_is_fp32, dout, lse, const_cast<float*>(p.delta), const_cast<float*>(p.lse2),
                                P->T, p.stat_pitch, P->Hq, P->D, P->D == 256 ? p.scale : 1.f, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  const size_t nq = (size_t)P->T * P->Hq * P->D, nk = (size_t)P->T * P->Hkv * P->D;
  e = cudaMemsetAsync(p.dq_acc, 0, nq * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.dk_acc, 0, nk * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.dv_acc, 0, nk * 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "accumulator reset");
  return RA_OK;
}

// One backward ring-step launch over work items [first, first + n) of the
// list at workspace offset `list`.
static ra_status bwd_step_launch(const ra_plan* P, size_t list, int64_t first, int64_t n, const void* q, const void* k,
                                 const void* v, const void* dout, void* dq, void* dk, void* dv, int32_t grads_fp32,
                                 void* workspace, const BwdLayout& L, void* stream_) {
  if (!q || !k || !v || !dout || (grads_fp32 && (!dq || !dk || !dv)))
    return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) ||
      (grads_fp32 && (!aligned16(dq) || !aligned16(dk) || !aligned16(dv))))
    return fail(RA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (n == 0) return RA_OK;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  ra::BwdParams p = bwd_params(P, L, ws, dq, dk, dv, grads_fp32);
  p.items = reinterpret_cast<const BwdItem*>(ws + list) + first;
  // head_dim 256: 64-row query tiles (with K and V resident, shared memory
  // holds one 64-row Q and dO tile)
  const int qrows = P->D == 256 ? 64 : 128;
  CUtensorMap tq, tk, tv, tdo, tl, td, tdq, tq64, tdo64;
  if (!encode_thd(&tq, q, P->T, P->Hq, P->D, qrows) || !encode_thd(&tk, k, P->T, P->Hkv, P->D) ||
      !encode_thd(&tv, v, P->T, P->Hkv, P->D) || !encode_thd(&tdo, dout, P->T, P->Hq, P->D, qrows) ||
      !encode_rows(&tl, p.lse2, p.stat_pitch, P->Hq, qrows) ||
      !encode_rows(&td, p.delta, p.stat_pitch, P->Hq, qrows) || !encode_acc(&tdq, p.dq_acc, P->T, P->Hq, P->D))
    return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor)");
  // CTA pairs: each CTA loads 64 of a query tile's 128 rows of Q and dO for S and dP
  if (bwd_pairs(*P) && (!encode_thd(&tq64, q, P->T, P->Hq, P->D, 64) || !encode_thd(&tdo64, dout, P->T, P->Hq, P->D, 64)))
    return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor)");
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = P->D == 256      ? ra::launch_bwd_step_d256(tq, tk, tv, tdo, tl, td, tdq, p, (int)n, st)
                  : bwd_pairs(*P) ? ra::launch_bwd_step_pair(tq, tq64, tk, tv, tdo, tdo64, tl, td, tdq, p, (int)n, st)
                                  : ra::launch_bwd_step(P->D, tq, tk, tv, tdo, tl, td, tdq, p, (int)n, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward step launch");
  return RA_OK;
}

ra_status ra_bwd_ring_step(const ra_plan* P, int32_t step, const void* q, const void* k, const void* v,
                           const void* dout, void* dq, void* dk, void* dv, int32_t grads_fp32, void* workspace,
                           size_t workspace_bytes, void* stream_) {
  BwdLayout L;
  ra_status rs = check_bwd_ws(P, grads_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (step < 0 || step >= P->steps) return fail(RA_ERR_INVALID_ARG, "step %d outside [0, %d)", step, P->steps);
  return bwd_step_launch(P, L.items, P->bwd_off[step], P->bwd_off[step + 1] - P->bwd_off[step], q, k, v, dout, dq,
                         dk, dv, grads_fp32, workspace, L, stream_);
}

ra_status ra_bwd_ring_step_rank(const ra_plan* P, int32_t step, int32_t rank, const void* q, const void* k,
                                const void* v, const void* dout, void* dq, void* dk, void* dv, int32_t grads_fp32,
                                void* workspace, size_t workspace_bytes, void* stream_) {
  BwdLayout L;
  ra_status rs = check_bwd_ws(P, grads_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (step < 0 || step >= P->steps) return fail(RA_ERR_INVALID_ARG, "step %d outside [0, %d)", step, P->steps);
  if (rank < 0 || rank >= P->steps) return fail(RA_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, P->steps);
  const int64_t c = (int64_t)step * P->steps + rank;
  return bwd_step_launch(P, L.ritems, P->bwd_rank_off[c], P->bwd_rank_off[c + 1] - P->bwd_rank_off[c], q, k, v, dout,
                         dq, dk, dv, grads_fp32, workspace, L, stream_);
}

ra_status ra_bwd_finish(const ra_plan* P, void* dq, void* dk, void* dv, int32_t grads_fp32, void* workspace,
                        size_t workspace_bytes, void* stream_) {
  BwdLayout L;
  ra_status rs = check_bwd_ws(P, grads_fp32, workspace, workspace_bytes, &L);
  if (rs != RA_OK) return rs;
  if (!dq || !dk || !dv || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RA_ERR_INVALID_ARG, "gradients must be 16-byte aligned device pointers");
  if (grads_fp32) return RA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const size_t nq = (size_t)P->T * P->Hq * P->D, nk = (size_t)P->T * P->Hkv * P->D;
  cudaError_t e = ra::launch_cast_bf16(reinterpret_cast<const float*>(ws + L.dq), dq, nq, st);
  if (e == cudaSuccess) e = ra::launch_cast_bf16(reinterpret_cast<const float*>(ws + L.dk), dk, nk, st);
  if (e == cudaSuccess) e = ra::launch_cast_bf16(reinterpret_cast<const float*>(ws + L.dv), dv, nk, st);
  if (e != cudaSuccess) return cuda_fail(e, "gradient cast launch");
  return RA_OK;
}

ra_status ra_bwd(const ra_plan* P, const void* q, const void* k, const void* v, const void* o, int32_t o_is_fp32,
                 const void* dout, const float* lse, void* dq, void* dk, void* dv, int32_t grads_fp32,
                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!P) return fail(RA_ERR_INVALID_ARG, "plan is NULL");
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return fail(RA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return fail(RA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  BwdLayout L;
  ra_status rs = check_bwd_ws(P, grads_fp32, workspace, workspace_bytes, &L);
  if (rs == RA_OK)
    rs = ra_bwd_prepare(P, o, o_is_fp32, dout, lse, dq, dk, dv, grads_fp32, workspace, workspace_bytes, stream);
  for (int32_t s = 0; s < P->steps && rs == RA_OK; ++s)
    rs = ra_bwd_ring_step(P, s, q, k, v, dout, dq, dk, dv, grads_fp32, workspace, workspace_bytes, stream);
  if (rs == RA_OK) rs = ra_bwd_finish(P, dq, dk, dv, grads_fp32, workspace, workspace_bytes, stream);
  return rs;
}

ra_status ra_selftest_wait_timeout(void* workspace, uint32_t limit_us, void* stream_) {
  if (!workspace || !aligned16(workspace)) return fail(RA_ERR_INVALID_ARG, "workspace must be a 16-byte aligned device pointer");
  if (limit_us < 1 || limit_us > 4000000) return fail(RA_ERR_INVALID_ARG, "limit_us must be in [1, 4000000]");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemsetAsync(workspace, 0, kHeader, st);
  if (e == cudaSuccess) e = ra::launch_wait_timeout_probe(reinterpret_cast<int*>(workspace), (uint64_t)limit_us * 1000u,
                                                          kSelfTestSite, st);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return RA_OK;
}

ra_status ra_workspace_status(const void* workspace, void* stream_) {
  if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word != 0) return fail(RA_ERR_TIMEOUT, "a kernel gave up on a pipeline wait (site %d)", word);
  return RA_OK;
}

}  // extern "C"
