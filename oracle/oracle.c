/*
 * oracle.c -- CPU oracle for one Medusa tree-speculative verify step.
 *
 * TEST INFRASTRUCTURE ONLY: see oracle.h.  Plain loops, double accumulation,
 * one thread.  Each function follows the definition it cites; nothing here is
 * blocked, fused or reordered for speed.
 */
#include "oracle.h"

#include <math.h>
#include <float.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element access                                                           */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t orc_bf16_round(double x) {
  /* Round to the nearest value with 8 significant bits (ties to even); that
   * value is exactly representable in binary32, whose top 16 bits are then
   * the bfloat16 encoding. */
  if (isnan(x)) return 0x7fc0;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs(x);
  double r;
  if (a == 0.0) {
    r = 0.0;
  } else if (isinf(a)) {
    r = INFINITY;
  } else {
    int e;
    (void)frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    if (e - 1 < -126) {
      /* subnormal range of bfloat16: quantum 2^-133 */
      r = ldexp(nearbyint(ldexp(a, 133)), -133);
    } else {
      r = ldexp(nearbyint(ldexp(a, 8 - e)), e - 8);
    }
    if (r > (double)FLT_MAX) r = INFINITY;
  }
  float f = (float)(neg ? -r : r);
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

double orc_load(const void* p, int dt, int64_t i) {
  if (dt == ORC_BF16) return bf16_to_double(((const uint16_t*)p)[i]);
  return (double)((const float*)p)[i];
}

void orc_store(void* p, int dt, int64_t i, double x) {
  if (dt == ORC_BF16)
    ((uint16_t*)p)[i] = orc_bf16_round(x);
  else
    ((float*)p)[i] = (float)x;
}

static double round_dt(int dt, double x) {
  if (dt == ORC_BF16) return bf16_to_double(orc_bf16_round(x));
  return (double)(float)x;
}

/* ------------------------------------------------------------------------ */
/* candidate tree                                                           */
/* ------------------------------------------------------------------------ */

/* Lexicographic order on rank paths; a proper prefix comes first. */
static int path_lex_cmp(const int32_t* a, int la, const int32_t* b, int lb) {
  int n = la < lb ? la : lb;
  for (int i = 0; i < n; ++i) {
    if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
  }
  if (la != lb) return la < lb ? -1 : 1;
  return 0;
}

/* Breadth-first order: depth first, then lexicographic. */
static int path_bfs_cmp(const int32_t* a, int la, const int32_t* b, int lb) {
  if (la != lb) return la < lb ? -1 : 1;
  return path_lex_cmp(a, la, b, lb);
}

int orc_tree_compile(const int32_t* paths, const int32_t* path_len, int n_paths,
                     int max_depth, int32_t* node_paths, int32_t* parent,
                     int32_t* depth, int32_t* rank, uint8_t* anc, int32_t* s,
                     int32_t* K_out) {
  if (n_paths < 0 || max_depth < 1) return -1;
  int T = n_paths + 1;
  /* order[] holds path indices sorted breadth-first (selection sort: the
   * plainest correct sort; trees are small). */
  int* order = (int*)malloc(sizeof(int) * (size_t)(n_paths > 0 ? n_paths : 1));
  for (int i = 0; i < n_paths; ++i) {
    if (path_len[i] < 1 || path_len[i] > max_depth) { free(order); return -1; }
    for (int j = 0; j < path_len[i]; ++j)
      if (paths[(int64_t)i * max_depth + j] < 1) { free(order); return -1; }
    order[i] = i;
  }
  for (int i = 0; i < n_paths; ++i) {
    int best = i;
    for (int j = i + 1; j < n_paths; ++j) {
      if (path_bfs_cmp(paths + (int64_t)order[j] * max_depth, path_len[order[j]],
                       paths + (int64_t)order[best] * max_depth,
                       path_len[order[best]]) < 0)
        best = j;
    }
    int t = order[i]; order[i] = order[best]; order[best] = t;
  }
  memset(node_paths, 0, sizeof(int32_t) * (size_t)T * max_depth);
  depth[0] = 0; parent[0] = -1; rank[0] = 0;
  for (int n = 1; n < T; ++n) {
    int src = order[n - 1];
    depth[n] = path_len[src];
    for (int j = 0; j < depth[n]; ++j)
      node_paths[(int64_t)n * max_depth + j] = paths[(int64_t)src * max_depth + j];
    rank[n] = node_paths[(int64_t)n * max_depth + depth[n] - 1];
  }
  /* duplicates */
  for (int n = 2; n < T; ++n)
    if (path_bfs_cmp(node_paths + (int64_t)n * max_depth, depth[n],
                     node_paths + (int64_t)(n - 1) * max_depth, depth[n - 1]) == 0) {
      free(order); return -1;
    }
  /* parent = the node whose path is this path minus its last rank */
  for (int n = 1; n < T; ++n) {
    parent[n] = -1;
    for (int m = 0; m < T; ++m) {
      if (depth[m] == depth[n] - 1 &&
          path_lex_cmp(node_paths + (int64_t)m * max_depth, depth[m],
                       node_paths + (int64_t)n * max_depth, depth[n] - 1) == 0) {
        parent[n] = m;
        break;
      }
    }
    if (parent[n] < 0) { free(order); return -1; }
  }
  /* ancestor-or-self: node m's path is a prefix of node n's path */
  for (int n = 0; n < T; ++n)
    for (int m = 0; m < T; ++m) {
      int is_anc = depth[m] <= depth[n] &&
                   path_lex_cmp(node_paths + (int64_t)m * max_depth, depth[m],
                                node_paths + (int64_t)n * max_depth, depth[m]) == 0;
      anc[(int64_t)n * T + m] = (uint8_t)is_anc;
    }
  int K = 0;
  for (int k = 0; k < max_depth; ++k) s[k] = 0;
  for (int n = 1; n < T; ++n) {
    if (depth[n] > K) K = depth[n];
    if (rank[n] > s[depth[n] - 1]) s[depth[n] - 1] = rank[n];
  }
  if (K_out) *K_out = K;
  free(order);
  return T;
}

int orc_tree_cartesian(const int32_t* s, int K, int max_nodes, int32_t* paths,
                       int32_t* path_len) {
  if (K < 1 || max_nodes < 0) return -1;
  int n = 0;
  int32_t idx[64];
  if (K > 64) return -1;
  /* depth by depth; within a depth, odometer order = lexicographic order */
  for (int k = 1; k <= K && n < max_nodes; ++k) {
    int any = 1;
    for (int j = 0; j < k; ++j) { idx[j] = 1; if (s[j] < 1) any = 0; }
    while (any && n < max_nodes) {
      for (int j = 0; j < K; ++j) paths[(int64_t)n * K + j] = j < k ? idx[j] : 0;
      path_len[n] = k;
      ++n;
      int j = k - 1;
      while (j >= 0) {
        if (idx[j] < s[j]) { ++idx[j]; break; }
        idx[j] = 1;
        --j;
      }
      if (j < 0) break;
    }
  }
  return n;
}

int orc_tree_greedy(const double* acc, int K, int R, int budget, int32_t* paths,
                    int32_t* path_len) {
  if (K < 1 || R < 1 || budget < 0 || K > 64) return -1;
  int n = 0;
  int32_t cand[64];
  int32_t best[64];
  while (n < budget) {
    double best_la = -INFINITY;
    int best_len = 0;
    int found = 0;
    /* every parent already in the tree (the root plus added nodes) */
    for (int p = -1; p < n; ++p) {
      int plen = p < 0 ? 0 : path_len[p];
      if (plen >= K) continue;
      for (int r = 1; r <= R; ++r) {
        for (int j = 0; j < plen; ++j) cand[j] = paths[(int64_t)p * K + j];
        cand[plen] = r;
        int clen = plen + 1;
        /* already added? */
        int dup = 0;
        for (int m = 0; m < n && !dup; ++m)
          if (path_lex_cmp(paths + (int64_t)m * K, path_len[m], cand, clen) == 0) dup = 1;
        if (dup) continue;
        double la = 0.0;
        for (int j = 0; j < clen; ++j) la += log(acc[(int64_t)j * R + (cand[j] - 1)]);
        int better;
        if (!found) better = 1;
        else if (la > best_la + 1e-9) better = 1;
        else if (la < best_la - 1e-9) better = 0;
        else better = path_lex_cmp(cand, clen, best, best_len) < 0;
        if (better) {
          found = 1;
          best_la = la;
          best_len = clen;
          for (int j = 0; j < clen; ++j) best[j] = cand[j];
        }
      }
    }
    if (!found) break;
    for (int j = 0; j < K; ++j) paths[(int64_t)n * K + j] = j < best_len ? best[j] : 0;
    path_len[n] = best_len;
    ++n;
  }
  return n;
}

double orc_tree_expected_len(const int32_t* paths, const int32_t* path_len,
                             int n_paths, int max_depth, const double* acc,
                             int R) {
  double e = 1.0; /* the root token is always emitted */
  for (int i = 0; i < n_paths; ++i) {
    double a = 1.0;
    for (int j = 0; j < path_len[i]; ++j)
      a *= acc[(int64_t)j * R + (paths[(int64_t)i * max_depth + j] - 1)];
    e += a;
  }
  return e;
}

/* ------------------------------------------------------------------------ */
/* rotary position embedding                                                */
/* ------------------------------------------------------------------------ */

void orc_rope(double* x, int Dh, int64_t pos, double theta) {
  int half = Dh / 2;
  for (int i = 0; i < half; ++i) {
    float inv_freq = (float)(1.0 / pow(theta, (2.0 * i) / (double)Dh));
    float ang = (float)pos * inv_freq;
    double c = cos((double)ang), s = sin((double)ang);
    double x1 = x[i], x2 = x[i + half];
    x[i] = x1 * c - x2 * s;
    x[i + half] = x2 * c + x1 * s;
  }
}

/* ------------------------------------------------------------------------ */
/* attention                                                                */
/* ------------------------------------------------------------------------ */

void orc_attn_one(int n, int Dh, const double* q, const double* k,
                  const double* v, double scale, double* out) {
  double* sc = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double d = 0.0;
    for (int t = 0; t < Dh; ++t) d += q[t] * k[(int64_t)j * Dh + t];
    sc[j] = d * scale;
    if (sc[j] > mx) mx = sc[j];
  }
  double den = 0.0;
  for (int j = 0; j < n; ++j) { sc[j] = exp(sc[j] - mx); den += sc[j]; }
  for (int t = 0; t < Dh; ++t) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += sc[j] * v[(int64_t)j * Dh + t];
    out[t] = n > 0 ? acc / den : 0.0;
  }
  free(sc);
}

int orc_tree_attn(int dt, const void* q, const void* k_new, const void* v_new,
                  void* k_cache, void* v_cache, const int64_t* seq_start,
                  const int32_t* prefix_len, const int32_t* depth,
                  const uint8_t* anc, int T, int B, int H, int Dh,
                  double rope_theta, double scale, void* out, double* out_d) {
  if (T < 1 || B < 1 || H < 1 || Dh < 2 || (Dh & 1)) return -1;
  const int64_t HD = (int64_t)H * Dh;
  double* x = (double*)malloc(sizeof(double) * (size_t)Dh);
  double* o = (double*)malloc(sizeof(double) * (size_t)Dh);
  /* 1. rotate the new keys at position L + depth and append K, V after the
   *    prefix: tree row i lives in slot L + i. */
  for (int b = 0; b < B; ++b) {
    const int64_t L = prefix_len[b];
    const int64_t st = seq_start[b];
    for (int i = 0; i < T; ++i) {
      for (int h = 0; h < H; ++h) {
        const int64_t src = (((int64_t)b * T + i) * H + h) * Dh;
        const int64_t dst = (st + L + i) * HD + (int64_t)h * Dh;
        for (int t = 0; t < Dh; ++t) x[t] = orc_load(k_new, dt, src + t);
        orc_rope(x, Dh, L + depth[i], rope_theta);
        for (int t = 0; t < Dh; ++t) orc_store(k_cache, dt, dst + t, x[t]);
        for (int t = 0; t < Dh; ++t)
          orc_store(v_cache, dt, dst + t, orc_load(v_new, dt, src + t));
      }
    }
  }
  /* 2. each row attends to the whole prefix and to its ancestors-or-self. */
  for (int b = 0; b < B; ++b) {
    const int64_t L = prefix_len[b];
    const int64_t st = seq_start[b];
    int nmax = (int)L + T;
    double* kk = (double*)malloc(sizeof(double) * (size_t)nmax * Dh);
    double* vv = (double*)malloc(sizeof(double) * (size_t)nmax * Dh);
    for (int i = 0; i < T; ++i) {
      for (int h = 0; h < H; ++h) {
        const int64_t qi = (((int64_t)b * T + i) * H + h) * Dh;
        for (int t = 0; t < Dh; ++t) x[t] = orc_load(q, dt, qi + t);
        orc_rope(x, Dh, L + depth[i], rope_theta);
        int n = 0;
        for (int64_t j = 0; j < L + T; ++j) {
          if (j >= L && !anc[(int64_t)i * T + (j - L)]) continue;
          const int64_t ki = (st + j) * HD + (int64_t)h * Dh;
          for (int t = 0; t < Dh; ++t) {
            kk[(int64_t)n * Dh + t] = orc_load(k_cache, dt, ki + t);
            vv[(int64_t)n * Dh + t] = orc_load(v_cache, dt, ki + t);
          }
          ++n;
        }
        orc_attn_one(n, Dh, x, kk, vv, scale, o);
        for (int t = 0; t < Dh; ++t) {
          orc_store(out, dt, qi + t, o[t]);
          if (out_d) out_d[qi + t] = o[t];
        }
      }
    }
    free(kk);
    free(vv);
  }
  free(x);
  free(o);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* LM head                                                                  */
/* ------------------------------------------------------------------------ */

int orc_lm_head(int dt, const void* hidden, const void* w, int rows, int d,
                int V, double* logits) {
  if (rows < 0 || d < 1 || V < 1) return -1;
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  for (int r = 0; r < rows; ++r) {
    for (int i = 0; i < d; ++i) h[i] = orc_load(hidden, dt, (int64_t)r * d + i);
    for (int v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += orc_load(w, dt, (int64_t)v * d + i) * h[i];
      logits[(int64_t)r * V + v] = acc;
    }
  }
  free(h);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* acceptance                                                               */
/* ------------------------------------------------------------------------ */

int orc_accept(const float* logits, const int32_t* tokens,
               const int32_t* parent, const int32_t* depth, int T, int K,
               int B, int V, int mode, double temperature, double eps,
               double delta, int32_t* accept_len, int32_t* accepted_nodes,
               int32_t* next_root, int32_t* best_node, double* best_logp,
               double* row_gap, double* node_margin, double* node_logp) {
  if (T < 1 || B < 1 || V < 1 || K < 0) return -1;
  if (mode != 0 && mode != 1) return -1;
  if (mode == 1 && !(temperature > 0.0)) return -1;
  int* amax = (int*)malloc(sizeof(int) * (size_t)T);
  double* mrow = (double*)malloc(sizeof(double) * (size_t)T);
  double* lse = (double*)malloc(sizeof(double) * (size_t)T);
  double* ent = (double*)malloc(sizeof(double) * (size_t)T);
  int* ok = (int*)malloc(sizeof(int) * (size_t)T);
  double* lp = (double*)malloc(sizeof(double) * (size_t)T);
  for (int b = 0; b < B; ++b) {
    /* per-row statistics of the backbone's prediction at each node */
    for (int p = 0; p < T; ++p) {
      const float* z = logits + ((int64_t)b * T + p) * V;
      int a = 0;
      for (int v = 1; v < V; ++v)
        if (z[v] > z[a]) a = v; /* first index among equal maxima */
      amax[p] = a;
      double second = -INFINITY;
      for (int v = 0; v < V; ++v)
        if (v != a && (double)z[v] > second) second = (double)z[v];
      if (row_gap) row_gap[(int64_t)b * T + p] = (double)z[a] - second;
      if (mode == 1) {
        /* p-hat = softmax(z / temperature); H = -sum p-hat log p-hat */
        double m = -INFINITY;
        for (int v = 0; v < V; ++v) {
          double y = (double)z[v] / temperature;
          if (y > m) m = y;
        }
        double S = 0.0;
        for (int v = 0; v < V; ++v) S += exp((double)z[v] / temperature - m);
        double logS = log(S) + m; /* log-sum-exp */
        double H = 0.0;
        for (int v = 0; v < V; ++v) {
          double lpv = (double)z[v] / temperature - logS;
          H -= exp(lpv) * lpv;
        }
        mrow[p] = m;
        lse[p] = logS;
        ent[p] = H;
      }
    }
    /* walk the tree breadth-first: a node is on an accepted prefix iff its
     * parent is and its own token passes the rule at the parent's row. */
    ok[0] = 1;
    lp[0] = 0.0;
    if (node_margin) node_margin[(int64_t)b * T] = 0.0;
    for (int c = 1; c < T; ++c) {
      int p = parent[c];
      int tok = tokens[(int64_t)b * T + c];
      int acc;
      double lpc = -INFINITY;
      if (mode == 0) {
        acc = (tok == amax[p]);
        if (node_margin) node_margin[(int64_t)b * T + c] = acc ? 1.0 : -1.0;
      } else {
        if (tok < 0 || tok >= V) {
          acc = 0;
          if (node_margin) node_margin[(int64_t)b * T + c] = -1.0;
        } else {
          const float* z = logits + ((int64_t)b * T + p) * V;
          lpc = (double)z[tok] / temperature - lse[p];
          double pr = exp(lpc);
          double thr = fmin(eps, delta * exp(-ent[p]));
          acc = pr > thr;
          if (node_margin) node_margin[(int64_t)b * T + c] = pr - thr;
        }
      }
      ok[c] = acc && ok[p];
      lp[c] = lp[p] + (mode == 1 ? lpc : 0.0);
    }
    if (node_logp)
      for (int c = 0; c < T; ++c) node_logp[(int64_t)b * T + c] = ok[c] ? lp[c] : -INFINITY;
    /* longest accepted prefix; typical ties by summed log-prob; then lowest
     * node index */
    int best = 0;
    for (int c = 1; c < T; ++c) {
      if (!ok[c]) continue;
      if (depth[c] > depth[best]) best = c;
      else if (depth[c] == depth[best] && mode == 1 && lp[c] > lp[best]) best = c;
    }
    accept_len[b] = depth[best];
    for (int j = 0; j <= K; ++j) accepted_nodes[(int64_t)b * (K + 1) + j] = -1;
    for (int c = best; c >= 0; c = parent[c])
      accepted_nodes[(int64_t)b * (K + 1) + depth[c]] = c;
    next_root[b] = amax[best];
    if (best_node) best_node[b] = best;
    if (best_logp) best_logp[b] = mode == 1 ? lp[best] : 0.0;
  }
  free(amax); free(mrow); free(lse); free(ent); free(ok); free(lp);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* KV compaction                                                            */
/* ------------------------------------------------------------------------ */

int orc_kv_compact(int dt, void* k_cache, void* v_cache,
                   const int64_t* seq_start, int32_t* prefix_len,
                   const int32_t* accepted_nodes, const int32_t* accept_len,
                   int B, int H, int Dh, int K, int32_t* src_slots) {
  if (B < 1 || H < 1 || Dh < 1 || K < 0) return -1;
  const int64_t HD = (int64_t)H * Dh;
  size_t esz = dt == ORC_BF16 ? 2 : 4;
  unsigned char* tk = (unsigned char*)malloc(esz * (size_t)(K + 1) * HD);
  unsigned char* tv = (unsigned char*)malloc(esz * (size_t)(K + 1) * HD);
  for (int b = 0; b < B; ++b) {
    const int64_t L = prefix_len[b];
    const int64_t st = seq_start[b];
    const int A = accept_len[b];
    if (A < 0 || A > K) { free(tk); free(tv); return -1; }
    /* read every source row first (a source may be a later destination) */
    for (int j = 0; j <= A; ++j) {
      int64_t a = accepted_nodes[(int64_t)b * (K + 1) + j];
      memcpy(tk + esz * j * HD, (unsigned char*)k_cache + esz * (st + L + a) * HD, esz * HD);
      memcpy(tv + esz * j * HD, (unsigned char*)v_cache + esz * (st + L + a) * HD, esz * HD);
    }
    for (int j = 0; j <= A; ++j) {
      memcpy((unsigned char*)k_cache + esz * (st + L + j) * HD, tk + esz * j * HD, esz * HD);
      memcpy((unsigned char*)v_cache + esz * (st + L + j) * HD, tv + esz * j * HD, esz * HD);
    }
    for (int j = 0; j <= K; ++j)
      src_slots[(int64_t)b * (K + 1) + j] =
          j <= A ? (int32_t)(L + accepted_nodes[(int64_t)b * (K + 1) + j]) : -1;
    prefix_len[b] = (int32_t)(L + A + 1);
  }
  free(tk);
  free(tv);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Medusa heads + top-s                                                     */
/* ------------------------------------------------------------------------ */

/* is (va, ia) ranked before (vb, ib)?  value descending, index ascending */
static int rank_before(double va, int ia, double vb, int ib) {
  if (va != vb) return va > vb;
  return ia < ib;
}

static void topk_double(const double* z, int V, int s, int32_t* out) {
  /* s passes of selection: the plainest full-sort-equivalent for small s */
  for (int j = 0; j < s; ++j) {
    int best = -1;
    for (int v = 0; v < V; ++v) {
      int taken = 0;
      for (int t = 0; t < j; ++t) if (out[t] == v) { taken = 1; break; }
      if (taken) continue;
      if (best < 0 || rank_before(z[v], v, z[best], best)) best = v;
    }
    out[j] = best;
  }
}

int orc_topk_f32(const float* z, int V, int s, int32_t* out) {
  if (V < 1 || s < 0 || s > V) return -1;
  double* zd = (double*)malloc(sizeof(double) * (size_t)V);
  for (int v = 0; v < V; ++v) zd[v] = (double)z[v];
  topk_double(zd, V, s, out);
  free(zd);
  return 0;
}

int orc_heads(int dt, const void* hidden, const int32_t* last_node, int T,
              const void* w1, const void* b1, const void* w2, const int32_t* s,
              int K, int B, int d, int V, double* head_logits, int32_t* topk,
              int s_max, void* u_out) {
  if (B < 1 || K < 1 || d < 1 || V < 1 || T < 1 || s_max < 0) return -1;
  for (int k = 0; k < K; ++k) if (s[k] < 0 || s[k] > s_max || s[k] > V) return -1;
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  double* u = (double*)malloc(sizeof(double) * (size_t)d);
  for (int b = 0; b < B; ++b) {
    int n = last_node[b];
    if (n < 0 || n >= T) { free(h); free(u); return -1; }
    for (int i = 0; i < d; ++i) h[i] = orc_load(hidden, dt, ((int64_t)b * T + n) * d + i);
    for (int k = 0; k < K; ++k) {
      int32_t* tk = topk + ((int64_t)b * K + k) * s_max;
      for (int j = 0; j < s_max; ++j) tk[j] = -1;
      if (s[k] == 0) continue;
      /* residual block: u = SiLU(W1 h + b1) + h, rounded to the weights'
       * type before the vocabulary projection */
      for (int j = 0; j < d; ++j) {
        double y = 0.0;
        for (int i = 0; i < d; ++i)
          y += orc_load(w1, dt, ((int64_t)k * d + j) * d + i) * h[i];
        if (b1) y += orc_load(b1, dt, (int64_t)k * d + j);
        double silu = y / (1.0 + exp(-y));
        u[j] = round_dt(dt, silu + h[j]);
        if (u_out) orc_store(u_out, dt, ((int64_t)b * K + k) * d + j, u[j]);
      }
      double* z = head_logits + ((int64_t)b * K + k) * V;
      for (int v = 0; v < V; ++v) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j)
          acc += orc_load(w2, dt, ((int64_t)k * V + v) * d + j) * u[j];
        z[v] = acc;
      }
      topk_double(z, V, s[k], tk);
    }
  }
  free(h);
  free(u);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* candidate fill                                                           */
/* ------------------------------------------------------------------------ */

int orc_build_candidates(const int32_t* next_root, const int32_t* topk,
                         int s_max, int K, const int32_t* depth,
                         const int32_t* rank, int T, int B, int32_t* tokens) {
  if (B < 1 || T < 1 || K < 0 || s_max < 1) return -1;
  for (int b = 0; b < B; ++b) {
    tokens[(int64_t)b * T] = next_root[b];
    for (int n = 1; n < T; ++n) {
      int k = depth[n] - 1, r = rank[n] - 1;
      if (k < 0 || k >= K || r < 0 || r >= s_max) return -1;
      tokens[(int64_t)b * T + n] = topk[((int64_t)b * K + k) * s_max + r];
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* rejection-sampling verification                                          */
/* ------------------------------------------------------------------------ */

double orc_rejection_emit(const double* p, const double* q, int n,
                          double* emitted) {
  /* accepted mass min(p,q); rejected mass (1-beta) re-drawn from the
   * normalised positive residual [p-q]_+ */
  double beta = 0.0;
  for (int x = 0; x < n; ++x) beta += fmin(p[x], q[x]);
  for (int x = 0; x < n; ++x) {
    double r = beta < 1.0 ? fmax(0.0, p[x] - q[x]) / (1.0 - beta) : 0.0;
    emitted[x] = fmin(p[x], q[x]) + (1.0 - beta) * r;
  }
  return beta;
}

/* softmax(z / tau) of one row, in double */
static void softmax_row(const float* z, int V, double tau, double* out) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) m = fmax(m, (double)z[v] / tau);
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    out[v] = exp((double)z[v] / tau - m);
    S += out[v];
  }
  for (int v = 0; v < V; ++v) out[v] /= S;
}

int orc_rejection_tree(const float* logits, const float* draft, const int32_t* tokens,
                       const int32_t* parent, const int32_t* depth, const int32_t* rank, int T,
                       int K, int B, int V, double temperature, const float* u, int u_stride,
                       int32_t* accept_len, int32_t* accepted_nodes, int32_t* next_token,
                       double* margin) {
  if (T < 1 || B < 1 || V < 1 || K < 0 || u_stride < 1 || !(temperature > 0.0)) return -1;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  int* kids = (int*)malloc(sizeof(int) * (size_t)T);
  for (int b = 0; b < B; ++b) {
    int cur = 0, len = 0;
    double mg = INFINITY;
    int32_t* an = accepted_nodes + (int64_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) an[j] = -1;
    an[0] = 0;
    softmax_row(logits + ((int64_t)b * T + 0) * V, V, temperature, p);
    int m = 0; /* children of the node where the walk stops */
    for (;;) {
      /* children of cur, in rank order */
      m = 0;
      for (int n = 0; n < T; ++n)
        if (n > 0 && parent[n] == cur) kids[m++] = n;
      for (int i = 1; i < m; ++i) /* insertion sort by rank */
        for (int j = i; j > 0 && rank[kids[j]] < rank[kids[j - 1]]; --j) {
          int t = kids[j]; kids[j] = kids[j - 1]; kids[j - 1] = t;
        }
      if (m == 0 || m >= u_stride) break;
      const int k = depth[kids[0]];
      if (k < 1 || k > K) break;
      softmax_row(draft + ((int64_t)b * K + (k - 1)) * V, V, temperature, q);
      int acc = -1;
      for (int j = 0; j < m; ++j) {
        const int n = kids[j];
        const int x = tokens[(int64_t)b * T + n];
        if (x < 0 || x >= V) continue; /* an invalid draft is never accepted */
        const double uu = (double)u[((int64_t)b * T + cur) * u_stride + j];
        const double lhs = uu * q[x], rhs = p[x];
        const double den = fmax(fmax(p[x], q[x]), 1e-300);
        mg = fmin(mg, fabs(lhs - rhs) / den);
        if (lhs < rhs) { acc = n; break; }
        /* rejected: the target becomes the normalised positive residual */
        double S = 0.0;
        for (int v = 0; v < V; ++v) S += fmax(0.0, p[v] - q[v]);
        if (S > 0.0)
          for (int v = 0; v < V; ++v) p[v] = fmax(0.0, p[v] - q[v]) / S;
      }
      if (acc < 0) break;
      an[++len] = acc;
      cur = acc;
      softmax_row(logits + ((int64_t)b * T + cur) * V, V, temperature, p);
    }
    /* the final token: inverse CDF of p at u[b][cur][m] */
    const int mm = m < u_stride ? m : u_stride - 1;
    const double uu = (double)u[((int64_t)b * T + cur) * u_stride + mm];
    double c = 0.0;
    int tok = -1;
    for (int v = 0; v < V; ++v) {
      if (p[v] <= 0.0) continue;
      const double c1 = c + p[v];
      if (tok < 0 && uu < c1) {
        tok = v;
        mg = fmin(mg, fmin(fabs(uu - c), fabs(c1 - uu)));
      }
      c = c1;
    }
    if (tok < 0) /* u beyond the rounded total: the last token with mass */
      for (int v = V - 1; v >= 0 && tok < 0; --v)
        if (p[v] > 0.0) tok = v;
    accept_len[b] = len;
    next_token[b] = tok;
    if (margin) margin[b] = mg;
  }
  free(p);
  free(q);
  free(kids);
  return 0;
}
