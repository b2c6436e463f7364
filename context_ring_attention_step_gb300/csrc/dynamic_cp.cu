// dynamic_cp.cu -- host-side Dynamic-CP sizing: per-sequence context-parallel
// group sizes and their placement on the ranks, from a cost model quadratic in
// the sequence length (Dynamic-CP page, "Modelado del programador de datos";
// power-of-two group sizes: "Construccion de multiples grupos de contexto
// paralelo por rango"; a static size set by the longest sequence splits short
// sequences needlessly: "Necesidad de un enfoque dinamico").
//
// Group size of a sequence (dynamic mode): the smallest power of two that fits
// the per-rank token limit and leaves none of its ranks more than the balanced
// share of the batch's time (sum of time(L) / ranks).
//
// The page describes its solver only as a heuristic.  This one places the
// sequences longest (most expensive) first, each on the aligned group of its
// size (ranks [g c, (g + 1) c)) whose busiest rank ends least loaded, within
// the per-rank token limit; a sequence that fits no group moves to the next
// larger group size.  The result feeds ra_plan_create's cp_size_per_doc.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "ring_attn_internal.h"

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

double seq_time(int64_t L, int causal, double sec_per_pair, double sec_per_token) {
  const double pairs = causal ? (double)(L * (L + 1) / 2) : (double)(L * L);
  return sec_per_pair * pairs + sec_per_token * (double)L;
}

}  // namespace

extern "C" ra_status ra_dynamic_cp(const int32_t* doc_lengths, int32_t num_docs, int32_t num_ranks,
                                   int64_t max_tokens_per_rank, int32_t causal, double sec_per_pair,
                                   double sec_per_token, int32_t mode, int32_t* cp_per_doc, int32_t* first_rank,
                                   double* rank_load, int64_t* rank_tokens) {
  using ra::set_last_error;
  if (num_docs < 0 || (num_docs > 0 && !doc_lengths))
    return set_last_error(RA_ERR_INVALID_ARG, "doc_lengths is NULL or num_docs < 0");
  if (num_ranks < 1 || num_ranks > (1 << 20) || (num_ranks & (num_ranks - 1)))
    return set_last_error(RA_ERR_INVALID_ARG, "num_ranks must be a power of two in [1, 2^20]");
  if (max_tokens_per_rank < 1) return set_last_error(RA_ERR_INVALID_ARG, "max_tokens_per_rank must be >= 1");
  if (mode != RA_CP_DYNAMIC && mode != RA_CP_STATIC)
    return set_last_error(RA_ERR_INVALID_ARG, "mode must be RA_CP_DYNAMIC or RA_CP_STATIC");
  if (!(sec_per_pair >= 0.0) || !(sec_per_token >= 0.0))
    return set_last_error(RA_ERR_INVALID_ARG, "cost coefficients must be >= 0");
  if (num_docs > 0 && (!cp_per_doc || !first_rank))
    return set_last_error(RA_ERR_INVALID_ARG, "cp_per_doc / first_rank is NULL");
  for (int32_t i = 0; i < num_docs; ++i)
    if (doc_lengths[i] < 0) return set_last_error(RA_ERR_INVALID_ARG, "negative document length");

  // smallest power-of-two group size whose shard fits the per-rank limit
  std::vector<int32_t> base(num_docs, 1);
  for (int32_t i = 0; i < num_docs; ++i) {
    int32_t c = 1;
    while (c <= num_ranks && ceil_div(doc_lengths[i], c) > max_tokens_per_rank) c *= 2;
    if (c > num_ranks) return set_last_error(RA_ERR_INVALID_ARG, "a sequence exceeds the memory of all ranks");
    base[i] = c;
  }
  std::vector<double> t(num_docs);
  for (int32_t i = 0; i < num_docs; ++i) t[i] = seq_time(doc_lengths[i], causal, sec_per_pair, sec_per_token);
  if (mode == RA_CP_STATIC && num_docs > 0) {  // every sequence gets the longest one's group size
    const int32_t top = *std::max_element(base.begin(), base.end());
    std::fill(base.begin(), base.end(), top);
  } else {
    // and a group large enough that none of its ranks takes more than the
    // balanced share of the batch's time
    double total = 0.0;
    for (int32_t i = 0; i < num_docs; ++i) total += t[i];
    const double share = total / num_ranks;
    for (int32_t i = 0; i < num_docs; ++i)
      while (base[i] < num_ranks && t[i] / base[i] > share) base[i] *= 2;
  }
  std::vector<int32_t> order(num_docs);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return t[a] > t[b]; });

  std::vector<double> load(num_ranks, 0.0);
  std::vector<int64_t> tokens(num_ranks, 0);
  for (int32_t i : order) {
    int32_t c = base[i];
    int32_t best_g = -1;
    while (true) {
      const int64_t share = ceil_div(doc_lengths[i], c);
      double best_end = 0.0;
      for (int32_t g = 0; g < num_ranks / c; ++g) {
        bool fits = true;
        double busiest = 0.0;
        for (int32_t r = g * c; r < (g + 1) * c; ++r) {
          if (tokens[r] + share > max_tokens_per_rank) { fits = false; break; }
          busiest = std::max(busiest, load[r]);
        }
        if (!fits) continue;
        const double end = busiest + t[i] / c;
        if (best_g < 0 || end < best_end) { best_end = end; best_g = g; }
      }
      if (best_g >= 0) break;
      c *= 2;
      if (c > num_ranks) return set_last_error(RA_ERR_INVALID_ARG, "the batch does not fit the ranks' memory");
    }
    cp_per_doc[i] = c;
    first_rank[i] = best_g * c;
    const int64_t share = ceil_div(doc_lengths[i], c);
    for (int32_t r = best_g * c; r < (best_g + 1) * c; ++r) {
      load[r] += t[i] / c;
      tokens[r] += share;
    }
  }
  if (rank_load) std::copy(load.begin(), load.end(), rank_load);
  if (rank_tokens) std::copy(tokens.begin(), tokens.end(), rank_tokens);
  return RA_OK;
}
