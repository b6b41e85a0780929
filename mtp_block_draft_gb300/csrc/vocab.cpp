// Frequent-token list of the draft heads (host only): counts raised by prompt tokens and
// picks and halved once 1024 have been counted; listed are the tokens whose count reaches
// three quarters of the size-th largest, and the conversation's tokens (colibri
// speculative-decoding doc, the token-list paragraph; readings in dmtp_vocab.h).
#include <algorithm>
#include <new>
#include <vector>

#include "dmtp_vocab.h"

struct dmtp_vocab_list {
  int V, size;
  std::vector<int64_t> counts;
  std::vector<uint8_t> member, conv;
  int counted = 0;
  int listed = 0;
  int64_t rebuilds = 0, appended = 0, picks = 0, picks_in = 0;
  std::vector<int64_t> scratch;

  bool ids_ok(const int32_t* t, int64_t n) const {
    if (n < 0 || (n > 0 && !t)) return false;
    for (int64_t i = 0; i < n; ++i)
      if (t[i] < 0 || t[i] >= V) return false;
    return true;
  }

  void rebuild() {
    // count_last: the size-th largest count (0 when size >= V is not reached by counts)
    int64_t last = 0;
    const int k = std::min(size, V);
    std::copy(counts.begin(), counts.end(), scratch.begin());  // sized at creation
    std::nth_element(scratch.begin(), scratch.begin() + (k - 1), scratch.end(),
                     [](int64_t a, int64_t b) { return a > b; });
    last = scratch[k - 1];
    listed = 0;
    for (int t = 0; t < V; ++t) {
      member[t] = (4 * counts[t] >= 3 * last) || conv[t];
      listed += member[t];
    }
    ++rebuilds;
  }

  void count(int t) {
    ++counts[t];
    if (++counted == DMTP_VOCAB_HALVE_EVERY) {
      for (int64_t& c : counts) c /= 2;
      counted = 0;
      rebuild();
    }
  }
};

extern "C" {

int dmtp_vocab_create(int vocab, int size, dmtp_vocab_list** out) {
  if (!out) return DMTP_EINVAL;
  *out = nullptr;
  if (vocab < 1 || size < 0) return DMTP_EINVAL;
  dmtp_vocab_list* v = new (std::nothrow) dmtp_vocab_list();
  if (!v) return DMTP_ENOMEM;
  try {
    v->V = vocab;
    v->size = size ? size : DMTP_VOCAB_DEFAULT_SIZE;
    v->counts.assign(vocab, 0);
    v->scratch.assign(vocab, 0);  // rebuild() allocates nothing after creation
    v->member.assign(vocab, 1);  // before the first request: every token
    v->conv.assign(vocab, 0);
    v->listed = vocab;
  } catch (...) {
    delete v;
    return DMTP_ENOMEM;
  }
  *out = v;
  return DMTP_OK;
}

int dmtp_vocab_begin_request(dmtp_vocab_list* v, const int32_t* prompt, int64_t n,
                             int new_conversation) {
  if (!v || !v->ids_ok(prompt, n)) return DMTP_EINVAL;
  if (new_conversation) std::fill(v->conv.begin(), v->conv.end(), 0);
  for (int64_t i = 0; i < n; ++i) v->conv[prompt[i]] = 1;
  for (int64_t i = 0; i < n; ++i) v->count(prompt[i]);
  v->rebuild();
  return DMTP_OK;
}

int dmtp_vocab_picked(dmtp_vocab_list* v, const int32_t* tokens, int64_t n) {
  if (!v || !v->ids_ok(tokens, n)) return DMTP_EINVAL;
  for (int64_t i = 0; i < n; ++i) {
    const int t = tokens[i];
    ++v->picks;
    v->picks_in += v->member[t];
    v->count(t);
    v->conv[t] = 1;
    if (!v->member[t]) {
      v->member[t] = 1;
      ++v->listed;
      ++v->appended;
    }
  }
  return DMTP_OK;
}

int dmtp_vocab_ids(const dmtp_vocab_list* v, int32_t* ids, int* listed) {
  if (!v) return DMTP_EINVAL;
  if (ids) {
    int j = 0;
    for (int t = 0; t < v->V; ++t)
      if (v->member[t]) ids[j++] = t;
  }
  if (listed) *listed = v->listed;
  return DMTP_OK;
}

int dmtp_vocab_mask(const dmtp_vocab_list* v, uint8_t* mask) {
  if (!v || !mask) return DMTP_EINVAL;
  std::copy(v->member.begin(), v->member.end(), mask);
  return DMTP_OK;
}

int dmtp_vocab_counts(const dmtp_vocab_list* v, int64_t* counts) {
  if (!v || !counts) return DMTP_EINVAL;
  std::copy(v->counts.begin(), v->counts.end(), counts);
  return DMTP_OK;
}

int dmtp_vocab_stats_read(const dmtp_vocab_list* v, dmtp_vocab_stats* out) {
  if (!v || !out) return DMTP_EINVAL;
  out->vocab = v->V;
  out->listed = v->listed;
  out->counted = v->counted;
  out->rebuilds = v->rebuilds;
  out->appended = v->appended;
  out->picks = v->picks;
  out->picks_in = v->picks_in;
  return DMTP_OK;
}

void dmtp_vocab_free(dmtp_vocab_list* v) { delete v; }

}  // extern "C"
