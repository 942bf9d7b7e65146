/*
 * lora_oracle.c -- plain, slow, obviously correct CPU oracle for the SGMV LoRA
 * delta and its batch routing.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Sources it follows (web pages, by title and section):
 *   - "max.pipelines.lora.LoRAManagerV3" API page, sort_lora_batch() and
 *     get_lora_graph_inputs(): the batch is ordered by adapter id with base
 *     (id -1) last; consecutive same-adapter requests are grouped into the
 *     triple (lora_ids, grouped_offsets, end), truncated at the first base
 *     group; end is the number of LoRA-routed tokens.
 *   - "vLLM LoRA 实现深度解析" section 1 (LoRA math): h = W0 x + (alpha/r) B A x,
 *     A in R^{r x k}, B in R^{d x r}; section 6 (multi-LoRA routing):
 *     output += lora_b_stacked[slot] . lora_a_stacked[slot] . x;
 *     section 9 (memory layout): lora_a_stacked [max_loras, max_lora_rank, in],
 *     lora_b_stacked [max_loras, out, max_lora_rank].
 *   - "MAX max.pipelines.lora 模块解析", section on the load pipeline (QKV
 *     fusion): q/k/v A matrices are concatenated on the rank dimension and B on
 *     the output dimension.  Under that layout slice j's B rows multiply only
 *     rank columns [jR, (j+1)R) of the intermediate (block-diagonal reading).
 *
 * Arithmetic: every product and sum is formed in IEEE double from values that
 * were converted exactly from their storage type by the caller.  No blocking,
 * no reordering: for each row, the shrink sums over the input index in
 * increasing order and the expand sums over the rank index in increasing
 * order.  The result handed back is the unrounded double y_in + B.(A.x); the
 * caller decides how (and whether) to round it to the storage type.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math).
 * A second build adds -fopenmp: the listed rows are then shared out among
 * threads (each row is computed by one thread, in the same order as above),
 * so both builds return bit-identical results; the single-threaded build
 * ignores the pragmas.
 */
#include <limits.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the row loops below run on: 1 in the single-threaded build; in the
 * OpenMP build, n > 0 first sets the count.  No arithmetic depends on it. */
int oracle_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* Status codes of the oracle (independent of the library's own codes). */
enum {
  ORACLE_OK = 0,
  ORACLE_BAD_ARG = 1,   /* negative count, negative length, null pointer */
  ORACLE_BAD_SLOT = 2,  /* slot < -1 or slot >= max_num_loras */
  ORACLE_BAD_ROW = 3,   /* a requested row is not a LoRA-routed row */
  ORACLE_BAD_ROUTE = 4  /* routing triple inconsistent */
};

/* Sort key of a request: its slot id, with base requests (-1) placed after
 * every adapter (the API page: "base id -1 sorts last"). */
static long long sort_key(int slot) { return slot < 0 ? (long long)INT_MAX + 1 : (long long)slot; }

/*
 * oracle_build_routing: sort, then group into the routing triple.
 *
 *   perm[i]            index (into the caller's request arrays) of the i-th
 *                      request of the sorted batch.  Stable insertion sort,
 *                      ascending key, so equal slots keep arrival order.
 *   lora_ids[g]        slot of group g, g < *num_groups.
 *   grouped_offsets[g] first token row of group g in the sorted batch;
 *                      grouped_offsets[*num_groups] == *end.
 *   *end               number of LoRA-routed token rows (all rows before the
 *                      first base request of the sorted batch).
 *   *total_tokens      token rows in the whole batch, base rows included.
 *
 * Requests with zero tokens still open (or continue) their adapter's group.
 * Output arrays: perm[n_req], lora_ids[max_num_loras],
 * grouped_offsets[max_num_loras + 1].
 */
int oracle_build_routing(int n_req, const int* req_slot, const int* req_len, int max_num_loras,
                         int* perm, int* lora_ids, int* grouped_offsets, int* num_groups, int* end,
                         int* total_tokens) {
  if (n_req < 0 || max_num_loras < 0) return ORACLE_BAD_ARG;
  if (!perm || !lora_ids || !grouped_offsets || !num_groups || !end || !total_tokens) return ORACLE_BAD_ARG;
  if (n_req > 0 && (!req_slot || !req_len)) return ORACLE_BAD_ARG;
  long long total = 0;
  for (int i = 0; i < n_req; ++i) {
    if (req_len[i] < 0) return ORACLE_BAD_ARG;
    if (req_slot[i] < -1 || req_slot[i] >= max_num_loras) return ORACLE_BAD_SLOT;
    total += req_len[i];
  }
  if (total > INT_MAX) return ORACLE_BAD_ARG;

  /* Stable insertion sort of request indices by key. */
  for (int i = 0; i < n_req; ++i) perm[i] = i;
  for (int i = 1; i < n_req; ++i) {
    int cur = perm[i];
    int j = i - 1;
    while (j >= 0 && sort_key(req_slot[perm[j]]) > sort_key(req_slot[cur])) {
      perm[j + 1] = perm[j];
      --j;
    }
    perm[j + 1] = cur;
  }

  /* Walk the sorted batch; a new group starts whenever the slot changes;
   * the walk stops at the first base request. */
  int g = 0;
  int row = 0;
  grouped_offsets[0] = 0;
  for (int i = 0; i < n_req; ++i) {
    int slot = req_slot[perm[i]];
    if (slot < 0) break;
    if (g == 0 || lora_ids[g - 1] != slot) {
      lora_ids[g] = slot;
      grouped_offsets[g] = row;
      ++g;
    }
    row += req_len[perm[i]];
    grouped_offsets[g] = row;
  }
  *num_groups = g;
  *end = row;
  *total_tokens = (int)total;
  return ORACLE_OK;
}

/* One projection slice of a (possibly fused) LoRA problem, all values double.
 *   A element (slot s, rank row k, input i): A[s*A_slot_stride + k*in_dim + i]
 *   B element (slot s, output o, rank k):    B[s*B_slot_stride + o*R + k]
 *   y_in / y_out element (listed row r, output o): y[r*row_stride + o]
 * For the fused q/k/v layout the caller points slice j at
 *   A_fused + j*R*in_dim (slot stride n*R*in_dim) and
 *   B_fused + off_j*R    (slot stride O*R),
 * which is exactly the block-diagonal reading of the fused weights.
 * An optional LoRA bias (the BIAS type of the MAX page's LoRA types; vLLM's
 * --enable-lora-bias) adds bias[s, o] to every routed output. */
typedef struct {
  const double* A;
  long long A_slot_stride;
  const double* B;
  long long B_slot_stride;
  int out_dim;
  const double* y_in;
  long long y_in_row_stride;
  double* y_out;
  long long y_out_row_stride;
  const double* bias;        /* bias of slot s, output o: bias[s*bias_slot_stride + o]; NULL: none */
  long long bias_slot_stride;
} oracle_slice;

/* Group of a LoRA-routed row, by linear scan of the offsets. */
static int group_of_row(int t, const int* grouped_offsets, int num_groups) {
  for (int g = 0; g < num_groups; ++g)
    if (grouped_offsets[g] <= t && t < grouped_offsets[g + 1]) return g;
  return -1;
}

/*
 * oracle_sgmv_rows: the LoRA delta for the listed token rows.
 *
 * rows[r] is the batch row t of the r-th listed row; x_rows, y_in and y_out
 * hold the listed rows only (row r of each belongs to batch row rows[r]).
 * For each listed row with 0 <= t < end, group g (grouped_offsets[g] <= t <
 * grouped_offsets[g+1]) and slot s = lora_ids[g], and for every slice j:
 *     u[r, j*R + k]   = sum_i A_j[s, k, i] * x_rows[r, i]              (k < R)
 *     y_out_j[r, o]   = y_in_j[r, o] + bias_j[s, o] + sum_k B_j[s, o, k] * u[r, j*R + k]
 * (bias term only when the slice has a bias).  u may be NULL.  A row t >= end (a base or post-end row) is an error: the
 * method never touches those rows, so the oracle refuses to produce them.
 */
int oracle_sgmv_rows(int n_rows, const int* rows, int in_dim, int R, int max_num_loras,
                     int n_slices, const oracle_slice* slices, const double* x_rows,
                     long long x_row_stride, const int* lora_ids, const int* grouped_offsets,
                     int num_groups, int end, double* u) {
  if (n_rows < 0 || in_dim <= 0 || R <= 0 || n_slices <= 0 || num_groups < 0) return ORACLE_BAD_ARG;
  if (n_rows > 0 && (!rows || !slices || !x_rows || !lora_ids || !grouped_offsets)) return ORACLE_BAD_ARG;
  if (num_groups > 0 && grouped_offsets[0] != 0) return ORACLE_BAD_ROUTE;
  for (int g = 0; g < num_groups; ++g) {
    if (grouped_offsets[g + 1] < grouped_offsets[g]) return ORACLE_BAD_ROUTE;
    if (lora_ids[g] < 0 || lora_ids[g] >= max_num_loras) return ORACLE_BAD_SLOT;
  }
  if (num_groups > 0 && grouped_offsets[num_groups] != end) return ORACLE_BAD_ROUTE;
  if (num_groups == 0 && end != 0) return ORACLE_BAD_ROUTE;

  if (R > 1024) return ORACLE_BAD_ARG;
  for (int r = 0; r < n_rows; ++r) {
    int t = rows[r];
    if (t < 0 || t >= end) return ORACLE_BAD_ROW;
    if (group_of_row(t, grouped_offsets, num_groups) < 0) return ORACLE_BAD_ROW;
  }

#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    int t = rows[r];
    int g = group_of_row(t, grouped_offsets, num_groups);
    int s = lora_ids[g];
    const double* xt = x_rows + (long long)r * x_row_stride;
    for (int j = 0; j < n_slices; ++j) {
      const oracle_slice* sl = &slices[j];
      /* shrink: u_j = A_j[s] . x_t */
      double uj[1024];
      for (int k = 0; k < R; ++k) {
        const double* a = sl->A + (long long)s * sl->A_slot_stride + (long long)k * in_dim;
        double acc = 0.0;
        for (int i = 0; i < in_dim; ++i) acc += a[i] * xt[i];
        uj[k] = acc;
        if (u) u[(long long)r * n_slices * R + (long long)j * R + k] = acc;
      }
      /* expand: y_j[t] = y_j[t] + B_j[s] . u_j */
      const double* yi = sl->y_in + (long long)r * sl->y_in_row_stride;
      double* yo = sl->y_out + (long long)r * sl->y_out_row_stride;
      for (int o = 0; o < sl->out_dim; ++o) {
        const double* b = sl->B + (long long)s * sl->B_slot_stride + (long long)o * R;
        double acc = 0.0;
        for (int k = 0; k < R; ++k) acc += b[k] * uj[k];
        const double bias = sl->bias ? sl->bias[(long long)s * sl->bias_slot_stride + o] : 0.0;
        yo[o] = yi[o] + bias + acc;
      }
    }
  }
  return ORACLE_OK;
}

/*
 * oracle_sgmv_token_slots: the delta defined per token, with no routing
 * triple ("vLLM LoRA 实现深度解析" section 6: token_lora_mapping gives the slot of
 * every token; output += lora_b_stacked[slot] . lora_a_stacked[slot] . x).
 * For each listed row r with slot row_slot[r] >= 0, and every slice j:
 *     u[r, j*R + k] = sum_i A_j[slot, k, i] * x_rows[r, i]
 *     y_out_j[r, o] = y_in_j[r, o] + sum_k B_j[slot, o, k] * u[r, j*R + k]
 * Rows with slot -1 (base) are copied unchanged to y_out and get u = 0.
 */
int oracle_sgmv_token_slots(int n_rows, const int* row_slot, int in_dim, int R, int max_num_loras,
                            int n_slices, const oracle_slice* slices, const double* x_rows,
                            long long x_row_stride, double* u) {
  if (n_rows < 0 || in_dim <= 0 || R <= 0 || R > 1024 || n_slices <= 0) return ORACLE_BAD_ARG;
  if (n_rows > 0 && (!row_slot || !slices || !x_rows)) return ORACLE_BAD_ARG;
  for (int r = 0; r < n_rows; ++r)
    if (row_slot[r] < -1 || row_slot[r] >= max_num_loras) return ORACLE_BAD_SLOT;
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    const int s = row_slot[r];
    const double* xt = x_rows + (long long)r * x_row_stride;
    for (int j = 0; j < n_slices; ++j) {
      const oracle_slice* sl = &slices[j];
      const double* yi = sl->y_in + (long long)r * sl->y_in_row_stride;
      double* yo = sl->y_out + (long long)r * sl->y_out_row_stride;
      if (s < 0) {
        for (int o = 0; o < sl->out_dim; ++o) yo[o] = yi[o];
        if (u)
          for (int k = 0; k < R; ++k) u[(long long)r * n_slices * R + (long long)j * R + k] = 0.0;
        continue;
      }
      double uj[1024];
      for (int k = 0; k < R; ++k) {
        const double* a = sl->A + (long long)s * sl->A_slot_stride + (long long)k * in_dim;
        double acc = 0.0;
        for (int i = 0; i < in_dim; ++i) acc += a[i] * xt[i];
        uj[k] = acc;
        if (u) u[(long long)r * n_slices * R + (long long)j * R + k] = acc;
      }
      for (int o = 0; o < sl->out_dim; ++o) {
        const double* b = sl->B + (long long)s * sl->B_slot_stride + (long long)o * R;
        double acc = 0.0;
        for (int k = 0; k < R; ++k) acc += b[k] * uj[k];
        const double bias = sl->bias ? sl->bias[(long long)s * sl->bias_slot_stride + o] : 0.0;
        yo[o] = yi[o] + bias + acc;
      }
    }
  }
  return ORACLE_OK;
}

/*
 * oracle_base_rows: the base projection of the listed rows ("vLLM LoRA
 * 实现深度解析" section 1: h = W0 x + (alpha/r) B A x; this is the W0 x term),
 *     y[r, o] = sum_i W0[o, i] * x_rows[r, i]        (o < out_dim)
 * in double, summing over the input index in increasing order.  W0 is the
 * projection's weight [out_dim, in_dim] (row o at W0 + o * w0_row_stride).
 * Its result is the y_in that oracle_sgmv_rows adds the delta to when the
 * delta is fused into the base projection.
 */
int oracle_base_rows(int n_rows, int in_dim, int out_dim, const double* W0, long long w0_row_stride,
                     const double* x_rows, long long x_row_stride, double* y, long long y_row_stride) {
  if (n_rows < 0 || in_dim <= 0 || out_dim <= 0) return ORACLE_BAD_ARG;
  if (n_rows > 0 && (!W0 || !x_rows || !y)) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    const double* xt = x_rows + (long long)r * x_row_stride;
    double* yr = y + (long long)r * y_row_stride;
    for (int o = 0; o < out_dim; ++o) {
      const double* w = W0 + (long long)o * w0_row_stride;
      double acc = 0.0;
      for (int i = 0; i < in_dim; ++i) acc += w[i] * xt[i];
      yr[o] = acc;
    }
  }
  return ORACLE_OK;
}
