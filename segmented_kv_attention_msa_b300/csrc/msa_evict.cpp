// Host-side KV-block eviction policy of AsymCache (paper "Multi-Segment Attention:
// Enabling Efficient KV-Cache Management for Faster Large Language Model Serving":
// abstract -- eviction that weighs hit rate against position-aware recompute cost;
// Fig. 6 / Eq. 5 -- marginal recompute latency of a block; Fig. 7 / Fig. 8 -- reuse-time
// distribution and a piecewise exponential reuse model, kept in an O(log n) structure;
// Fig. 10 / Eq. 10 -- the lambda update from the mean block lifespan; appendix A.1 --
// only an exponential keeps the order of untouched blocks).
//
// Score of a cached block b at time t (evict the smallest):
//   S_b(t) = C_b * min(1, lambda * F_b * exp(-(t - t_b) / beta))
//   C_b    = k5 * p_b + (k2 - k3 + k5)      Eq. 5 with (l1 + 2 q1) approximated by p_b,
//                                           the number of blocks before b in its sequence
//   F_b    = accesses of b while cached;  t_b = its last access
//   lambda = exp((tau - tau0) / beta - tau / alpha)   Eq. 10, tau = mean lifespan
//            (eviction time - insertion time) over the last `window` evictions, refreshed
//            every `period` evictions
// The reuse estimate is flat (1) until the turning point t_b + beta * ln(lambda F_b) and
// decays exponentially after it.  Scaling F by lambda moves every turning point by
// beta * ln(lambda).
//
// Ordered structure: with kappa_b = ln F_b + t_b / beta and theta(t) = t / beta - ln lambda,
// a block is flat while kappa_b >= theta, with ln S = ln C_b, and decaying otherwise, with
// ln S = ln C_b + kappa_b - theta.  Within each class the order of two blocks that are not
// accessed never changes (the decay is exponential), so each class is kept in ordered sets
// keyed by time-independent values; blocks cross between classes as theta moves.  Every
// operation is O(log n).  A linear-scan mode computes the same scores directly (O(n) per
// eviction), and LRU and prefix-only orders serve as baselines.
#include <stdint.h>

#include <cmath>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "msa.h"

namespace {

struct Block {
  double lnC;      // ln C_b
  double kappa;    // ln F_b + t_b / beta
  double t_last;   // last access
  double t_ins;    // insertion
  int32_t pos;     // p_b
  int32_t count;   // F_b
  bool flat;
};

using Key = std::pair<double, int32_t>;  // (value, block id): ties go to the smaller id

}  // namespace

struct msa_evict {
  msa_evict_opts_t o;
  double ln_lambda;
  std::unordered_map<int32_t, Block> blocks;
  // cost-aware policy: flat class by (ln C) and by (kappa); decaying class by (ln C + kappa)
  // and by (kappa)
  std::set<Key> flat_c, flat_k, dec_s, dec_k;
  // baselines: LRU by (last access); prefix-only by (-position, last access)
  std::set<std::pair<double, int32_t>> lru;
  std::set<std::pair<std::pair<int32_t, double>, int32_t>> prefix;
  std::vector<double> life;  // lifespans of the last `window` evictions (ring)
  int32_t life_next = 0, life_n = 0, since_update = 0;
};

namespace {

inline double theta(const msa_evict* p, double t) { return t / p->o.beta - p->ln_lambda; }

void attach(msa_evict* p, int32_t id, Block& b, double t) {
  switch (p->o.policy) {
    case MSA_EVICT_COST:
      b.flat = b.kappa >= theta(p, t);
      if (b.flat) {
        p->flat_c.insert({b.lnC, id});
        p->flat_k.insert({b.kappa, id});
      } else {
        p->dec_s.insert({b.lnC + b.kappa, id});
        p->dec_k.insert({b.kappa, id});
      }
      break;
    case MSA_EVICT_LRU:
      p->lru.insert({b.t_last, id});
      break;
    case MSA_EVICT_PREFIX:
      p->prefix.insert({{-b.pos, b.t_last}, id});
      break;
    default:
      break;
  }
}

void detach(msa_evict* p, int32_t id, const Block& b) {
  switch (p->o.policy) {
    case MSA_EVICT_COST:
      if (b.flat) {
        p->flat_c.erase({b.lnC, id});
        p->flat_k.erase({b.kappa, id});
      } else {
        p->dec_s.erase({b.lnC + b.kappa, id});
        p->dec_k.erase({b.kappa, id});
      }
      break;
    case MSA_EVICT_LRU:
      p->lru.erase({b.t_last, id});
      break;
    case MSA_EVICT_PREFIX:
      p->prefix.erase({{-b.pos, b.t_last}, id});
      break;
    default:
      break;
  }
}

// Move blocks across the flat / decaying boundary for time t.
void migrate(msa_evict* p, double t) {
  const double th = theta(p, t);
  while (!p->flat_k.empty() && p->flat_k.begin()->first < th) {
    const int32_t id = p->flat_k.begin()->second;
    Block& b = p->blocks[id];
    p->flat_c.erase({b.lnC, id});
    p->flat_k.erase(p->flat_k.begin());
    b.flat = false;
    p->dec_s.insert({b.lnC + b.kappa, id});
    p->dec_k.insert({b.kappa, id});
  }
  while (!p->dec_k.empty() && std::prev(p->dec_k.end())->first >= th) {
    const auto it = std::prev(p->dec_k.end());
    const int32_t id = it->second;
    Block& b = p->blocks[id];
    p->dec_s.erase({b.lnC + b.kappa, id});
    p->dec_k.erase(it);
    b.flat = true;
    p->flat_c.insert({b.lnC, id});
    p->flat_k.insert({b.kappa, id});
  }
}

// ln S_b(t) straight from the definition.
double ln_score(const msa_evict* p, const Block& b, double t) {
  const double e = std::log((double)b.count) - (t - b.t_last) / p->o.beta + p->ln_lambda;
  return b.lnC + (e < 0.0 ? e : 0.0);
}

void record_lifespan(msa_evict* p, double span) {
  if (p->o.window <= 0) return;
  p->life[p->life_next] = span;
  p->life_next = (p->life_next + 1) % p->o.window;
  if (p->life_n < p->o.window) ++p->life_n;
  if (p->o.period > 0 && ++p->since_update >= p->o.period) {
    p->since_update = 0;
    double sum = 0.0;
    for (int32_t i = 0; i < p->life_n; ++i) sum += p->life[i];
    const double tau = sum / p->life_n;
    // Eq. 10, kept as ln lambda.  kappa does not depend on lambda, so no set is re-keyed:
    // the flat / decaying split moves at the next query (migrate).
    p->ln_lambda = (tau - p->o.tau0) / p->o.beta - tau / p->o.alpha;
  }
}

bool valid_opts(const msa_evict_opts_t* o) {
  if (!o) return false;
  if (!(o->beta > 0.0) || !(o->alpha > 0.0) || !(o->lambda0 > 0.0)) return false;
  if (!(o->k5 >= 0.0) || !(o->k_const > 0.0)) return false;
  if (o->window < 0 || o->period < 0 || (o->period > 0 && o->window == 0)) return false;
  if (o->policy < MSA_EVICT_COST || o->policy > MSA_EVICT_PREFIX) return false;
  return std::isfinite(o->tau0) && std::isfinite(o->k5) && std::isfinite(o->k_const);
}

}  // namespace

extern "C" msa_status_t msa_evict_create(const msa_evict_opts_t* opts, msa_evict_t** out) {
  if (!out) return MSA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!valid_opts(opts)) return MSA_ERR_INVALID_ARG;
  msa_evict* p = new (std::nothrow) msa_evict();
  if (!p) return MSA_ERR_INVALID_ARG;
  p->o = *opts;
  p->ln_lambda = std::log(opts->lambda0);
  p->life.assign((size_t)opts->window, 0.0);
  *out = p;
  return MSA_OK;
}

extern "C" void msa_evict_destroy(msa_evict_t* p) { delete p; }

extern "C" msa_status_t msa_evict_insert(msa_evict_t* p, int32_t block, int32_t pos_block, double now) {
  if (!p || block < 0 || pos_block < 0 || !std::isfinite(now)) return MSA_ERR_INVALID_ARG;
  if (p->blocks.count(block)) return MSA_ERR_INVALID_ARG;
  Block b;
  b.pos = pos_block;
  b.count = 1;
  b.t_last = now;
  b.t_ins = now;
  b.lnC = std::log(p->o.k5 * (double)pos_block + p->o.k_const);
  b.kappa = now / p->o.beta;  // ln 1 + t_b / beta
  b.flat = true;
  Block& slot = p->blocks[block];
  slot = b;
  attach(p, block, slot, now);
  return MSA_OK;
}

extern "C" msa_status_t msa_evict_access(msa_evict_t* p, int32_t block, double now) {
  if (!p || !std::isfinite(now)) return MSA_ERR_INVALID_ARG;
  auto it = p->blocks.find(block);
  if (it == p->blocks.end()) return MSA_ERR_INVALID_ARG;
  Block& b = it->second;
  detach(p, block, b);
  b.count += 1;
  b.t_last = now;
  b.kappa = std::log((double)b.count) + now / p->o.beta;
  attach(p, block, b, now);
  return MSA_OK;
}

extern "C" msa_status_t msa_evict_remove(msa_evict_t* p, int32_t block) {
  if (!p) return MSA_ERR_INVALID_ARG;
  auto it = p->blocks.find(block);
  if (it == p->blocks.end()) return MSA_ERR_INVALID_ARG;
  detach(p, block, it->second);
  p->blocks.erase(it);
  return MSA_OK;
}

extern "C" msa_status_t msa_evict_victim(msa_evict_t* p, double now, int32_t* block) {
  if (!p || !block || !std::isfinite(now)) return MSA_ERR_INVALID_ARG;
  *block = -1;
  if (p->blocks.empty()) return MSA_ERR_INVALID_ARG;
  int32_t id = -1;
  switch (p->o.policy) {
    case MSA_EVICT_COST: {
      migrate(p, now);
      const double th = theta(p, now);
      bool have = false;
      Key best{0.0, 0};
      if (!p->flat_c.empty()) {
        best = *p->flat_c.begin();
        have = true;
      }
      if (!p->dec_s.empty()) {
        const Key d{p->dec_s.begin()->first - th, p->dec_s.begin()->second};
        if (!have || d < best) best = d;
        have = true;
      }
      id = best.second;
      break;
    }
    case MSA_EVICT_COST_SCAN: {
      Key best{INFINITY, -1};
      for (const auto& kv : p->blocks) {
        const Key k{ln_score(p, kv.second, now), kv.first};
        if (best.second < 0 || k < best) best = k;
      }
      id = best.second;
      break;
    }
    case MSA_EVICT_LRU:
      id = p->lru.begin()->second;
      break;
    case MSA_EVICT_PREFIX:
      id = p->prefix.begin()->second;
      break;
    default:
      return MSA_ERR_INVALID_ARG;
  }
  auto it = p->blocks.find(id);
  const double span = now - it->second.t_ins;
  detach(p, id, it->second);
  p->blocks.erase(it);
  record_lifespan(p, span);
  *block = id;
  return MSA_OK;
}

extern "C" msa_status_t msa_evict_score(const msa_evict_t* p, int32_t block, double now, double* score) {
  if (!p || !score) return MSA_ERR_INVALID_ARG;
  auto it = p->blocks.find(block);
  if (it == p->blocks.end()) return MSA_ERR_INVALID_ARG;
  *score = std::exp(ln_score(p, it->second, now));
  return MSA_OK;
}

extern "C" msa_status_t msa_evict_get_lambda(const msa_evict_t* p, double* lambda) {
  if (!p || !lambda) return MSA_ERR_INVALID_ARG;
  *lambda = std::exp(p->ln_lambda);
  return MSA_OK;
}

extern "C" int32_t msa_evict_size(const msa_evict_t* p) { return p ? (int32_t)p->blocks.size() : 0; }

extern "C" msa_status_t msa_evict_check(const msa_evict_t* p, double now) {
  // structural self-check for tests: every block sits in exactly the sets of its class
  if (!p) return MSA_ERR_INVALID_ARG;
  if (p->o.policy == MSA_EVICT_COST) {
    if (p->flat_c.size() != p->flat_k.size() || p->dec_s.size() != p->dec_k.size()) return MSA_ERR_INVALID_ARG;
    if (p->flat_c.size() + p->dec_s.size() != p->blocks.size()) return MSA_ERR_INVALID_ARG;
    for (const auto& kv : p->blocks) {
      const Block& b = kv.second;
      if (b.flat ? !p->flat_c.count({b.lnC, kv.first}) || !p->flat_k.count({b.kappa, kv.first})
                 : !p->dec_s.count({b.lnC + b.kappa, kv.first}) || !p->dec_k.count({b.kappa, kv.first}))
        return MSA_ERR_INVALID_ARG;
    }
    (void)now;
  } else if (p->o.policy == MSA_EVICT_LRU) {
    if (p->lru.size() != p->blocks.size()) return MSA_ERR_INVALID_ARG;
  } else if (p->o.policy == MSA_EVICT_PREFIX) {
    if (p->prefix.size() != p->blocks.size()) return MSA_ERR_INVALID_ARG;
  }
  return MSA_OK;
}
