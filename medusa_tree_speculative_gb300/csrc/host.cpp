// Host side of libmedusa: error reporting, device queries and the candidate
// tree helpers ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads", Method items 2-4).  No CUDA kernels here.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <vector>

#include "internal.h"

namespace medusa {

static thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MEDUSA_OK;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

int check_tree(const medusa_tree_t* t, const char* what) {
  if (!t) return fail(MEDUSA_ERR_INVALID, "%s: tree is NULL", what);
  if (t->T < 1 || t->T > MEDUSA_MAX_T)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: tree T=%d outside [1, %d]", what, t->T, MEDUSA_MAX_T);
  if (t->W != (t->T + 31) / 32) return fail(MEDUSA_ERR_INVALID, "%s: tree W=%d != ceil(T/32)", what, t->W);
  if (t->K < 0 || t->K > MEDUSA_MAX_K)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: tree depth K=%d outside [0, %d]", what, t->K, MEDUSA_MAX_K);
  if ((t->T > 1) != (t->K > 0)) return fail(MEDUSA_ERR_INVALID, "%s: tree T=%d with depth %d", what, t->T, t->K);
  if (!t->parent || !t->depth || !t->rank || !t->anc_mask)
    return fail(MEDUSA_ERR_INVALID, "%s: tree has a NULL device array", what);
  for (int k = 0; k < t->K; ++k)
    if (t->s[k] < 1 || t->s[k] > MEDUSA_MAX_S)
      return fail(MEDUSA_ERR_INVALID, "%s: tree s[%d]=%d outside [1, %d]", what, k, t->s[k], MEDUSA_MAX_S);
  return MEDUSA_OK;
}

}  // namespace medusa

using namespace medusa;

extern "C" const char* medusa_last_error(void) { return g_last_error; }
extern "C" const char* medusa_version(void) { return "libmedusa 0.1 (sm_103a)"; }

// --------------------------------------------------------------------------
// Candidate tree helpers
// --------------------------------------------------------------------------

namespace {
using Path = std::vector<int32_t>;

// breadth-first: shorter first, then lexicographic
bool bfs_less(const Path& a, const Path& b) {
  if (a.size() != b.size()) return a.size() < b.size();
  return std::lexicographical_compare(a.begin(), a.end(), b.begin(), b.end());
}
}  // namespace

extern "C" int medusa_tree_compile(const int32_t* paths, const int32_t* path_len, int n_paths,
                                   int max_depth, int32_t* parent, int32_t* depth, int32_t* rank,
                                   uint32_t* anc_mask, int32_t* s, int32_t* node_paths, int* T_out,
                                   int* K_out) {
  if (n_paths < 0 || max_depth < 1 || (n_paths > 0 && (!paths || !path_len)) || !parent || !depth ||
      !rank || !anc_mask || !s || !T_out || !K_out)
    return fail(MEDUSA_ERR_INVALID, "medusa_tree_compile: bad argument");
  const int T = n_paths + 1;
  if (T > MEDUSA_MAX_T) return fail(MEDUSA_ERR_UNSUPPORTED, "medusa_tree_compile: %d rows > %d", T, MEDUSA_MAX_T);
  std::vector<Path> all;
  all.reserve(T);
  all.push_back(Path());  // the root
  for (int i = 0; i < n_paths; ++i) {
    int len = path_len[i];
    if (len < 1 || len > max_depth)
      return fail(MEDUSA_ERR_INVALID, "medusa_tree_compile: path %d has length %d", i, len);
    if (len > MEDUSA_MAX_K)
      return fail(MEDUSA_ERR_UNSUPPORTED, "medusa_tree_compile: depth %d > %d", len, MEDUSA_MAX_K);
    Path p(paths + (size_t)i * max_depth, paths + (size_t)i * max_depth + len);
    for (int32_t r : p) {
      if (r < 1) return fail(MEDUSA_ERR_INVALID, "medusa_tree_compile: path %d has rank %d", i, r);
      if (r > MEDUSA_MAX_S)
        return fail(MEDUSA_ERR_UNSUPPORTED, "medusa_tree_compile: rank %d > %d", r, MEDUSA_MAX_S);
    }
    all.push_back(std::move(p));
  }
  std::sort(all.begin() + 1, all.end(), bfs_less);
  std::map<Path, int> index;
  for (int n = 0; n < T; ++n) {
    if (!index.emplace(all[n], n).second)
      return fail(MEDUSA_ERR_INVALID, "medusa_tree_compile: duplicate path");
  }
  const int W = (T + 31) / 32;
  std::memset(anc_mask, 0, sizeof(uint32_t) * (size_t)T * W);
  std::memset(s, 0, sizeof(int32_t) * (size_t)max_depth);
  int K = 0;
  for (int n = 0; n < T; ++n) {
    const Path& p = all[n];
    depth[n] = (int32_t)p.size();
    rank[n] = p.empty() ? 0 : p.back();
    if (n == 0) {
      parent[n] = -1;
    } else {
      auto it = index.find(Path(p.begin(), p.end() - 1));
      if (it == index.end()) return fail(MEDUSA_ERR_INVALID, "medusa_tree_compile: a path's prefix is missing");
      parent[n] = it->second;
      K = std::max(K, (int)p.size());
      s[p.size() - 1] = std::max(s[p.size() - 1], p.back());
    }
    // ancestor-or-self bits: follow the parent chain
    for (int a = n; a >= 0; a = parent[a]) anc_mask[(size_t)n * W + a / 32] |= 1u << (a % 32);
    if (node_paths) {
      for (int j = 0; j < max_depth; ++j) node_paths[(size_t)n * max_depth + j] = j < (int)p.size() ? p[j] : 0;
    }
  }
  *T_out = T;
  *K_out = K;
  return MEDUSA_OK;
}

extern "C" int medusa_tree_cartesian(const int32_t* s, int K, int max_nodes, int32_t* paths,
                                     int32_t* path_len) {
  if (!s || K < 1 || K > MEDUSA_MAX_K || max_nodes < 0 || (max_nodes > 0 && (!paths || !path_len)))
    return fail(MEDUSA_ERR_INVALID, "medusa_tree_cartesian: bad argument");
  int n = 0;
  long long level = 1;
  for (int k = 1; k <= K && n < max_nodes; ++k) {
    if (s[k - 1] < 1) break;
    level *= s[k - 1];
    // node number m at this depth, written in mixed radix (s_1, ..., s_k),
    // is the path in lexicographic order
    for (long long m = 0; m < level && n < max_nodes; ++m) {
      long long rem = m;
      for (int j = k - 1; j >= 0; --j) {
        paths[(size_t)n * K + j] = (int32_t)(rem % s[j]) + 1;
        rem /= s[j];
      }
      for (int j = k; j < K; ++j) paths[(size_t)n * K + j] = 0;
      path_len[n] = k;
      ++n;
    }
  }
  return n;
}

extern "C" int medusa_tree_greedy(const double* acc, int K, int R, int budget, int32_t* paths,
                                  int32_t* path_len) {
  if (!acc || K < 1 || K > MEDUSA_MAX_K || R < 1 || budget < 0 || (budget > 0 && (!paths || !path_len)))
    return fail(MEDUSA_ERR_INVALID, "medusa_tree_greedy: bad argument");
  struct Cand {
    Path p;
    double logacc;
  };
  std::vector<Cand> frontier;
  auto push_children = [&](const Path& parent_path, double parent_logacc) {
    if ((int)parent_path.size() >= K) return;
    const int k = (int)parent_path.size();
    for (int r = 1; r <= R; ++r) {
      Cand c{parent_path, parent_logacc + std::log(acc[(size_t)k * R + (r - 1)])};
      c.p.push_back(r);
      frontier.push_back(std::move(c));
    }
  };
  push_children(Path(), 0.0);
  int n = 0;
  while (n < budget && !frontier.empty()) {
    size_t best = 0;
    for (size_t i = 1; i < frontier.size(); ++i) {
      const double d = frontier[i].logacc - frontier[best].logacc;
      if (d > 1e-9 || (std::fabs(d) <= 1e-9 && std::lexicographical_compare(
                                                   frontier[i].p.begin(), frontier[i].p.end(),
                                                   frontier[best].p.begin(), frontier[best].p.end())))
        best = i;
    }
    Cand c = std::move(frontier[best]);
    frontier.erase(frontier.begin() + (long)best);
    for (int j = 0; j < K; ++j) paths[(size_t)n * K + j] = j < (int)c.p.size() ? c.p[j] : 0;
    path_len[n] = (int32_t)c.p.size();
    ++n;
    push_children(c.p, c.logacc);
  }
  return n;
}
