// tail.cuh -- the work done by the last CTA of an argmax launch once every
// row's argmax is known: greedy accept (verify), prefill commit, or a draft
// write. Header-only so each kernel file inlines it.
#pragma once
#include "common.cuh"

namespace spec {

// Runs in the last CTA of an argmax launch. best[] holds every pass row's
// packed argmax; it is consumed and zeroed here together with the counter.
__device__ __forceinline__ void run_tail(const TailArgs& t) {
  unsigned long long* best = t.best_all;
  const int b = threadIdx.x;
  if (t.mode == TAIL_VERIFY && b < t.B) {
    // Greedy accept ("Gemma 4's MTP drafter explained", section "How does
    // speculative decoding work?"): keep drafts up to the first one that
    // differs from the target's choice, then append the target's own token.
    const int slot = t.seq_ids[b], R = t.k + 1;
    int tok[17];
    for (int i = 0; i < R; ++i) tok[i] = (int)best_index(volatile_load(best + b * R + i));
    int A = 0;
    while (A < t.k && t.drafts[b * t.k + A] == tok[A]) ++A;
    for (int i = 0; i < R; ++i) t.out_tokens[b * R + i] = i <= A ? tok[i] : -1;
    t.n_emitted[b] = A + 1;
    const int err = t.err ? *(volatile int*)t.err : 0;
    if (!err) {
      t.seq_len[slot] += A + 1;
      t.pending[slot] = tok[A];
      t.stats[slot * 4 + 0] += 1;
      t.stats[slot * 4 + 1] += t.k;
      t.stats[slot * 4 + 2] += A;
      t.stats[slot * 4 + 3] += A + 1;
    }
    t.sel_row[b] = b * R + A;
  } else if (t.mode == TAIL_TREE && b < t.B) {
    // Tree verify: from the root (row 0, the pending token) the lowest-index
    // child node whose token is the target's choice at the current row is
    // accepted, then its children are tried, and so on; row r is node r - 1.
    const int slot = t.seq_ids[b], R = t.k + 1;
    int tok[17];
    for (int i = 0; i < R; ++i) tok[i] = (int)best_index(volatile_load(best + b * R + i));
    int cur = 0, A = 0;
    t.path[b * t.path_ld] = 0;
    for (;;) {
      int next = -1;
      for (int c = 0; c < t.k; ++c)
        if (t.parents[b * t.k + c] + 1 == cur && t.drafts[b * t.k + c] == tok[cur]) {
          next = c + 1;
          break;
        }
      if (next < 0) break;
      t.out_tokens[b * R + A] = t.drafts[b * t.k + next - 1];
      ++A;
      t.path[b * t.path_ld + A] = next;
      cur = next;
    }
    t.out_tokens[b * R + A] = tok[cur];
    for (int i = A + 1; i < R; ++i) t.out_tokens[b * R + i] = -1;
    t.n_emitted[b] = A + 1;
    const int err = t.err ? *(volatile int*)t.err : 0;
    if (!err) {
      t.seq_len[slot] += A + 1;
      t.pending[slot] = tok[cur];
      t.stats[slot * 4 + 0] += 1;
      t.stats[slot * 4 + 1] += t.k;
      t.stats[slot * 4 + 2] += A;
      t.stats[slot * 4 + 3] += A + 1;
    }
    t.sel_row[b] = b * R + cur;
  } else if (t.mode == TAIL_PREFILL && b < t.B) {
    const int slot = t.seq_ids[b], R = t.R;
    const int last = (int)best_index(volatile_load(best + b * R + R - 1));
    const int err = t.err ? *(volatile int*)t.err : 0;
    if (!err) {
      t.seq_len[slot] += R;
      t.pending[slot] = last;
    }
    t.sel_row[b] = b * R + R - 1;
  } else if (t.mode == TAIL_DRAFT && b < t.B) {
    int row = (int)best_index(volatile_load(best + b));
    t.draft_out[b * t.draft_ld + t.draft_j] = t.token_of ? t.token_of[row] : row;
  }
  __syncthreads();
  const int nrows = t.mode == TAIL_DRAFT ? t.B : t.B * (t.mode == TAIL_VERIFY || t.mode == TAIL_TREE ? t.k + 1 : t.R);
  for (int i = threadIdx.x; i < nrows; i += blockDim.x) best[i] = 0ull;
  if (threadIdx.x == 0) *t.counter = 0u;
}

}  // namespace spec
