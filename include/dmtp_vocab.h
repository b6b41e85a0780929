/*
 * dmtp_vocab.h — the frequent-token list the draft heads score instead of the whole
 * vocabulary.
 *
 * Source: colibri speculative-decoding doc, the paragraph on the token list a draft head
 * scores in place of the full vocabulary: the `size` most frequent tokens (16000 unless
 * set), any other token whose frequency reaches three quarters of the smallest
 * frequency among those, and the tokens of the conversation being served. Each prompt
 * token and each committed pick raises its token's count by one, and all counts are
 * halved once 1024 tokens have been counted since the last halving; the list is
 * recomputed at each request start and after each halving, and an unlisted pick is
 * added immediately. Verification still scores the full vocabulary, so the committed
 * tokens are unaffected. The DMTP blog (section 6.5) names shortlisting before exact
 * scoring as the next step for the T1 head.
 *
 * Readings where the page leaves a step open (the same in the test oracle): counts are
 * integers and halve by floor division; the 1024th counted token since the last halving
 * triggers it; the three-quarters rule is 4 count >= 3 count_last, count_last the size-th
 * largest count (so ties never change the list; with fewer than `size` counted tokens it
 * is 0 and every token is listed); a request start clears the conversation when asked,
 * joins the prompt's tokens to it, counts them in order (a halving in between rebuilds)
 * and rebuilds; a picked token is counted, joins the conversation and, if missing, the
 * list; one list may serve a whole batch (its conversation is the union). Before the
 * first request the list is the whole vocabulary.
 *
 * Host-only: no device memory, no CUDA calls; one caller at a time. Every int-returning
 * call returns DMTP_OK or a negative DMTP_E* code (dmtp.h); a call that fails (a token
 * id outside [0, vocab)) leaves the list unchanged.
 */
#ifndef DMTP_VOCAB_H
#define DMTP_VOCAB_H

#include <stdint.h>

#include "dmtp.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DMTP_VOCAB_DEFAULT_SIZE 16000
#define DMTP_VOCAB_HALVE_EVERY 1024

typedef struct dmtp_vocab_list dmtp_vocab_list; /* opaque, owned by the library */

typedef struct {
  int vocab;
  int listed;         /* tokens on the list now                          */
  int counted;        /* tokens counted since the last halving           */
  int64_t rebuilds;   /* request starts plus halvings                    */
  int64_t appended;   /* picked tokens that joined between rebuilds      */
  int64_t picks;      /* picked tokens counted                            */
  int64_t picks_in;   /* of those, already on the list when picked       */
} dmtp_vocab_stats;

/* A list over `vocab` (>= 1) tokens; size: the highest-count tokens kept (>= 1; 0 means
 * DMTP_VOCAB_DEFAULT_SIZE). */
int dmtp_vocab_create(int vocab, int size, dmtp_vocab_list** out);

/* A request starts: prompt = host array [n] of token ids (n >= 0; NULL when n = 0);
 * new_conversation != 0 clears the conversation first. */
int dmtp_vocab_begin_request(dmtp_vocab_list* v, const int32_t* prompt, int64_t n,
                             int new_conversation);

/* Tokens picked (committed), host array [n], in order. */
int dmtp_vocab_picked(dmtp_vocab_list* v, const int32_t* tokens, int64_t n);

/* The listed ids in increasing order into ids (host array [vocab], or NULL) and their
 * number into *listed (may be NULL). */
int dmtp_vocab_ids(const dmtp_vocab_list* v, int32_t* ids, int* listed);

/* mask[t] = 1 when token t is listed, else 0 (host array [vocab]). */
int dmtp_vocab_mask(const dmtp_vocab_list* v, uint8_t* mask);

/* The current counts (host array [vocab]). */
int dmtp_vocab_counts(const dmtp_vocab_list* v, int64_t* counts);

int dmtp_vocab_stats_read(const dmtp_vocab_list* v, dmtp_vocab_stats* out);

/* Never fails; NULL is a no-op. */
void dmtp_vocab_free(dmtp_vocab_list* v);

#ifdef __cplusplus
}
#endif
#endif /* DMTP_VOCAB_H */
