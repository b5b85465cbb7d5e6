/*
 * Seeded synthetic inputs for the KV residency path: row contents and
 * per-step sparse selections.  This module is shared by the CUDA path's
 * tests/bench and by the CPU oracle's tests; it holds none of the method's
 * arithmetic (no dedup, no mapping, no replacement policy) -- only random
 * numbers and the workload recipe.
 *
 * Random numbers: SplitMix64 as published by Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators" (OOPSLA 2014): a 64-bit
 * counter advanced by the golden-ratio gamma, followed by the variant-13
 * 64-bit finaliser.  Every stream is keyed by the fields it depends on, so
 * any row or selection can be regenerated independently of the others.
 *
 * Row contents stand for an FP8 MLA row (512 e4m3 latent bytes, 4 fp32
 * scales, 64 bf16 rope values = 656 bytes) and are uniform random bytes,
 * a pure function of (seed, group, layer, logical address).
 *
 * Selections follow the decode-step shape of index-based sparse attention
 * (UlaCache page, "Unified logical addresses" and "Experiments"): per
 * request and query token, top-k positions = the recent window, plus a
 * fraction kept from the previous selection, plus fresh positions drawn
 * from the rest of the history (uniform or Zipf over position).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYNTH_PAD 0xFFFFFFFFu

static inline uint64_t sm64_next(uint64_t *state) {
  uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* A stream state keyed by four fields: chain the fields through the mixer. */
static uint64_t sm64_key(uint64_t a, uint64_t b, uint64_t c, uint64_t d) {
  uint64_t s = a;
  uint64_t x = sm64_next(&s);
  s = x ^ b;
  x = sm64_next(&s);
  s = x ^ c;
  x = sm64_next(&s);
  s = x ^ d;
  return sm64_next(&s);
}

/* uniform integer in [0, n), n < 2^32: high 32 bits scaled (multiply-shift) */
static inline uint32_t sm64_below(uint64_t *s, uint32_t n) {
  return (uint32_t)(((sm64_next(s) >> 32) * (uint64_t)n) >> 32);
}

static inline double sm64_unit(uint64_t *s) {
  return (double)(sm64_next(s) >> 11) * (1.0 / 9007199254740992.0);
}

enum { DOMAIN_CONTENT = 0x636f6e74u, DOMAIN_SEL = 0x73656c65u, DOMAIN_CTX = 0x63747878u,
       DOMAIN_APPEND = 0x61707064u, DOMAIN_PAD = 0x70616464u };

/* ------------------------------------------------------------------ rows */

static void fill_row(uint64_t seed, uint32_t g, uint32_t j, uint32_t addr,
                     uint32_t row_bytes, uint8_t *dst) {
  uint64_t s = sm64_key(seed ^ ((uint64_t)DOMAIN_CONTENT << 32), g, j, addr);
  uint32_t b = 0;
  for (; b + 8 <= row_bytes; b += 8) {
    uint64_t x = sm64_next(&s);
#if defined(__BYTE_ORDER__) && __BYTE_ORDER__ == __ORDER_LITTLE_ENDIAN__
    memcpy(dst + b, &x, 8); /* the bytes of x, least significant first */
#else
    for (int i = 0; i < 8; ++i) dst[b + i] = (uint8_t)(x >> (8 * i));
#endif
  }
  if (b < row_bytes) {
    uint64_t x = sm64_next(&s);
    for (int i = 0; b < row_bytes; ++b, ++i) dst[b] = (uint8_t)(x >> (8 * i));
  }
}

/* out[n][L][row_bytes]: rows of layers 0..L-1 of group g for addresses addr0..addr0+n-1 */
void synth_content_range(uint64_t seed, uint32_t g, uint32_t L, uint32_t addr0, uint32_t n,
                         uint32_t row_bytes, uint8_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    for (uint32_t j = 0; j < L; ++j)
      fill_row(seed, g, j, addr0 + (uint32_t)i, row_bytes,
               out + ((size_t)i * L + j) * row_bytes);
}

/* out[n][row_bytes]: layer j of group g for an arbitrary address list (PAD rows are zero) */
void synth_content_list(uint64_t seed, uint32_t g, uint32_t j, const uint32_t *addrs, uint32_t n,
                        uint32_t row_bytes, uint8_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    if (addrs[i] == SYNTH_PAD)
      memset(out + (size_t)i * row_bytes, 0, row_bytes);
    else
      fill_row(seed, g, j, addrs[i], row_bytes, out + (size_t)i * row_bytes);
  }
}

/* -------------------------------------------------------------- selections */

typedef struct {
  uint64_t seed;
  uint32_t n_groups;        /* selection groups G (one independent selection each) */
  uint32_t n_live;          /* requests decoding at once (R) */
  uint32_t n_total;         /* requests over the whole trace (> n_live with turnover) */
  uint32_t ctx_min, ctx_max;/* initial context length, uniform integer in [min, max] */
  uint32_t q;               /* query tokens per request per step */
  uint32_t k;               /* top-k per query token */
  uint32_t window;          /* recent window always selected */
  double keep;              /* fraction of the non-window budget kept from the previous set */
  uint32_t fresh_zipf;      /* 0: fresh positions uniform; 1: Zipf over absolute position */
  double zipf_s;            /* Zipf exponent */
  uint32_t append_max;      /* tokens appended per request per step: uniform in [1, append_max]; 0 none */
  uint32_t append_cap;      /* cap on tokens appended per request */
  uint32_t turnover_period; /* every P steps the oldest request finishes and the next joins; 0 none */
  double pad_prob;          /* probability that an entry is replaced by the pad marker */
} synth_params;

typedef struct {
  uint32_t free_base, free_n;   /* logical range released after the step (n = 0: none) */
  uint32_t append_base, append_n;/* logical range allocated for appended tokens (n = 0: none) */
  uint32_t join_base, join_n;   /* logical range allocated for a joining request (n = 0: none) */
} synth_events;

typedef struct {
  uint32_t id;       /* global request id */
  uint32_t base;     /* first logical address of the initial context */
  uint32_t ctx0;     /* initial context length */
  uint32_t n_app;    /* appended tokens */
  uint32_t *app;     /* appended logical addresses [append_cap] */
  uint32_t steps;    /* steps this request has decoded */
  uint32_t *prev;    /* previous q0 selection per group: [G][k] positions */
  uint32_t *prev_n;  /* [G] */
} synth_req;

typedef struct {
  synth_params p;
  synth_req *live;      /* [n_live], oldest first */
  uint32_t next_req;    /* next request id to join */
  uint32_t next_logical;/* the library's monotonic logical-address counter, simulated */
  uint32_t step;
  uint32_t max_len;
  uint8_t *mark;        /* [max_len] scratch */
  uint32_t *cand;       /* [k] scratch */
  uint32_t *cur;        /* [k] scratch: the set being built */
  uint32_t *prevq;      /* [k] scratch: previous query token's set in this step */
  double *zipf_cdf;     /* [zipf_len] */
  uint32_t zipf_len;
} synth_trace;

static uint32_t draw_ctx(const synth_params *p, uint32_t id) {
  uint64_t s = sm64_key(p->seed ^ ((uint64_t)DOMAIN_CTX << 32), id, 0, 0);
  uint32_t span = p->ctx_max - p->ctx_min + 1;
  return p->ctx_min + (span ? sm64_below(&s, span) : 0);
}

static void req_init(synth_trace *t, synth_req *r, uint32_t id) {
  const synth_params *p = &t->p;
  r->id = id;
  r->ctx0 = draw_ctx(p, id);
  r->base = t->next_logical;
  t->next_logical += r->ctx0;
  r->n_app = 0;
  r->steps = 0;
  memset(r->prev_n, 0, sizeof(uint32_t) * p->n_groups);
}

static inline uint32_t req_len(const synth_req *r) { return r->ctx0 + r->n_app; }
static inline uint32_t req_addr(const synth_req *r, uint32_t pos) {
  return pos < r->ctx0 ? r->base + pos : r->app[pos - r->ctx0];
}

synth_trace *synth_trace_create(const synth_params *p) {
  if (!p || p->n_live == 0 || p->n_total < p->n_live || p->k == 0 || p->q == 0 ||
      p->ctx_min == 0 || p->ctx_max < p->ctx_min || p->n_groups == 0)
    return NULL;
  if (p->turnover_period && p->append_max) return NULL; /* finishing requests own one range */
  synth_trace *t = (synth_trace *)calloc(1, sizeof(synth_trace));
  t->p = *p;
  t->max_len = p->ctx_max + (p->append_max ? p->append_cap : 0);
  t->mark = (uint8_t *)calloc(t->max_len, 1);
  t->cand = (uint32_t *)malloc(sizeof(uint32_t) * p->k);
  t->cur = (uint32_t *)malloc(sizeof(uint32_t) * p->k);
  t->prevq = (uint32_t *)malloc(sizeof(uint32_t) * p->k);
  t->live = (synth_req *)calloc(p->n_live, sizeof(synth_req));
  for (uint32_t i = 0; i < p->n_live; ++i) {
    t->live[i].app = (uint32_t *)malloc(sizeof(uint32_t) * (p->append_cap + 1));
    t->live[i].prev = (uint32_t *)malloc(sizeof(uint32_t) * p->n_groups * p->k);
    t->live[i].prev_n = (uint32_t *)calloc(p->n_groups, sizeof(uint32_t));
    req_init(t, &t->live[i], i);
  }
  t->next_req = p->n_live;
  if (p->fresh_zipf) {
    t->zipf_len = 0; /* table built on first use */
    t->zipf_cdf = (double *)malloc(sizeof(double) * t->max_len);
  }
  return t;
}

void synth_trace_destroy(synth_trace *t) {
  if (!t) return;
  for (uint32_t i = 0; i < t->p.n_live; ++i) {
    free(t->live[i].app);
    free(t->live[i].prev);
    free(t->live[i].prev_n);
  }
  free(t->live);
  free(t->mark);
  free(t->cand);
  free(t->cur);
  free(t->prevq);
  free(t->zipf_cdf);
  free(t);
}

/* Initial context of every live request, in live order; logical ranges are
 * consecutive from 0 in that order.  Returns the number of logical addresses. */
uint32_t synth_trace_initial(const synth_trace *t, uint32_t *ctx_out, uint32_t *base_out) {
  for (uint32_t i = 0; i < t->p.n_live; ++i) {
    if (ctx_out) ctx_out[i] = t->live[i].ctx0;
    if (base_out) base_out[i] = t->live[i].base;
  }
  return t->next_logical;
}

/* Context length of request id (including ones that join later). */
uint32_t synth_request_ctx(const synth_params *p, uint32_t id) { return draw_ctx(p, id); }

static uint32_t zipf_draw(synth_trace *t, uint64_t *s, uint32_t len) {
  /* inverse CDF of P(p) ~ (p+1)^-s over p in [0, len); table rebuilt when len changes */
  if (t->zipf_len != len) {
    t->zipf_len = len;
    double acc = 0.0;
    for (uint32_t i = 0; i < len; ++i) {
      acc += pow((double)i + 1.0, -t->p.zipf_s);
      t->zipf_cdf[i] = acc;
    }
    for (uint32_t i = 0; i < len; ++i) t->zipf_cdf[i] /= acc;
  }
  double u = sm64_unit(s);
  uint32_t lo = 0, hi = len - 1;
  while (lo < hi) {
    uint32_t mid = lo + (hi - lo) / 2;
    if (t->zipf_cdf[mid] < u) lo = mid + 1; else hi = mid;
  }
  return lo;
}

/* Build one top-k position set for request r.  prev/prev_n: the set it
 * overlaps with (none for a request's first step).  Writes positions to
 * t->cur and returns how many (k unless the history is shorter than k). */
static uint32_t build_set(synth_trace *t, synth_req *r, uint64_t *s,
                          const uint32_t *prev, uint32_t prev_n) {
  const synth_params *p = &t->p;
  uint32_t len = req_len(r);
  uint32_t n = 0;
  if (len <= p->k) {
    for (uint32_t i = 0; i < len; ++i) t->cur[n++] = i;
    return n;
  }
  uint32_t wlen = p->window < len ? p->window : len;
  uint32_t wstart = len - wlen;
  for (uint32_t i = wstart; i < len; ++i) t->cur[n++] = i;
  uint32_t budget = p->k - wlen;
  uint32_t kept = 0;
  if (prev && prev_n) {
    uint32_t nc = 0;
    for (uint32_t i = 0; i < prev_n; ++i)
      if (prev[i] < wstart) t->cand[nc++] = prev[i];
    uint32_t want = (uint32_t)floor(p->keep * (double)budget);
    if (want > nc) want = nc;
    for (uint32_t i = 0; i < want; ++i) { /* partial Fisher-Yates */
      uint32_t j = i + sm64_below(s, nc - i);
      uint32_t tmp = t->cand[i]; t->cand[i] = t->cand[j]; t->cand[j] = tmp;
      t->cur[n++] = t->cand[i];
      t->mark[t->cand[i]] = 1;
    }
    kept = want;
  }
  uint32_t fresh = budget - kept;
  uint32_t room = wstart - kept; /* positions outside the window and not kept */
  if (fresh > room) fresh = room;
  while (fresh) {
    uint32_t pos = p->fresh_zipf ? zipf_draw(t, s, len) : sm64_below(s, wstart);
    if (pos >= wstart || t->mark[pos]) continue;
    t->mark[pos] = 1;
    t->cur[n++] = pos;
    --fresh;
  }
  for (uint32_t i = wlen; i < n; ++i) t->mark[t->cur[i]] = 0;
  return n;
}

/* One decode step: sel[G][n_live][q][k] logical addresses (PAD where the
 * history is shorter than k or a pad was injected), then the events that
 * follow the step (the caller applies them in this order: free, join,
 * appends; that is the order in which logical ranges were assigned). */
void synth_trace_step(synth_trace *t, uint32_t *sel, synth_events *ev) {
  const synth_params *p = &t->p;
  const size_t qk = (size_t)p->q * p->k;
  for (uint32_t g = 0; g < p->n_groups; ++g) {
    for (uint32_t ri = 0; ri < p->n_live; ++ri) {
      synth_req *r = &t->live[ri];
      uint32_t *dst = sel + ((size_t)g * p->n_live + ri) * qk;
      uint64_t s = sm64_key(p->seed ^ ((uint64_t)DOMAIN_SEL << 32), r->id,
                            ((uint64_t)r->steps << 8), g);
      uint64_t sp = sm64_key(p->seed ^ ((uint64_t)DOMAIN_PAD << 32), r->id, r->steps, g);
      uint32_t prevq_n = 0;
      for (uint32_t qi = 0; qi < p->q; ++qi) {
        const uint32_t *pv = qi == 0 ? r->prev + (size_t)g * p->k : t->prevq;
        uint32_t pn = qi == 0 ? (r->steps ? r->prev_n[g] : 0) : prevq_n;
        uint32_t n = build_set(t, r, &s, pv, pn);
        uint32_t *row = dst + (size_t)qi * p->k;
        for (uint32_t i = 0; i < n; ++i) row[i] = req_addr(r, t->cur[i]);
        for (uint32_t i = n; i < p->k; ++i) row[i] = SYNTH_PAD;
        if (p->pad_prob > 0.0)
          for (uint32_t i = 0; i < p->k; ++i)
            if (sm64_unit(&sp) < p->pad_prob) row[i] = SYNTH_PAD;
        memcpy(t->prevq, t->cur, sizeof(uint32_t) * n);
        prevq_n = n;
        if (qi == 0) {
          memcpy(r->prev + (size_t)g * p->k, t->cur, sizeof(uint32_t) * n);
          r->prev_n[g] = n;
        }
      }
    }
  }
  for (uint32_t ri = 0; ri < p->n_live; ++ri) t->live[ri].steps++;
  memset(ev, 0, sizeof(*ev));
  /* turnover: the oldest live request finishes, the next one joins */
  if (p->turnover_period && (t->step + 1) % p->turnover_period == 0 && t->next_req < p->n_total) {
    synth_req done = t->live[0];
    ev->free_base = done.base;
    ev->free_n = done.ctx0;
    memmove(&t->live[0], &t->live[1], sizeof(synth_req) * (p->n_live - 1));
    t->live[p->n_live - 1] = done; /* reuse its buffers */
    req_init(t, &t->live[p->n_live - 1], t->next_req++);
    ev->join_base = t->live[p->n_live - 1].base;
    ev->join_n = t->live[p->n_live - 1].ctx0;
  }
  /* appends: accepted tokens per request, allocated as one consecutive range in live order */
  if (p->append_max) {
    uint32_t base = t->next_logical, total = 0;
    for (uint32_t ri = 0; ri < p->n_live; ++ri) {
      synth_req *r = &t->live[ri];
      uint64_t s = sm64_key(p->seed ^ ((uint64_t)DOMAIN_APPEND << 32), r->id, t->step, 0);
      uint32_t a = 1 + sm64_below(&s, p->append_max);
      uint32_t room = p->append_cap - r->n_app;
      if (a > room) a = room;
      for (uint32_t i = 0; i < a; ++i) r->app[r->n_app++] = base + total + i;
      total += a;
    }
    t->next_logical += total;
    ev->append_base = base;
    ev->append_n = total;
  }
  t->step++;
}

uint32_t synth_trace_next_logical(const synth_trace *t) { return t->next_logical; }
