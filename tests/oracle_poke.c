/*
 * Test-only build of the CPU oracle with one extra entry point that writes a
 * single field of the pool's state directly.  The invariant checker
 * orc_check() never sees a bad state in a correct run, so the tests use this
 * setter to put one source into each state a check must reject and assert
 * that exactly that check fires.  Compiled by tests/test_oracle_check.py with
 * ORC_SOURCE set to the oracle source the oracle module builds (so a planted
 * mistake in that source is seen here too); nothing else links it.
 */
#include ORC_SOURCE

enum {
  POKE_TAG = 0,       /* tags[i] = v */
  POKE_STAMP = 1,     /* stamps[i] = v */
  POKE_PAGE_SLOT = 2, /* page_slot[i] = v */
  POKE_BACKED = 3,    /* backed[i] = v */
  POKE_PEND = 4,      /* pend[i] = v */
  POKE_SLOT_PAIR = 5, /* pool slot table: slot_pair[i] = v */
  POKE_SLOT_PAGE = 6, /* pool slot table: slot_page[i] = v */
  POKE_HOST = 7       /* host copy element i = v */
};

int orc_test_poke(orc_pool *p, int32_t r, int32_t s, int32_t field, int64_t i, int64_t v) {
  orc_source *src = get_src(p, r, s);
  if (!src || i < 0) return ORC_EINVAL;
  switch (field) {
    case POKE_TAG:
      if (i >= p->B) return ORC_EINVAL;
      src->tags[i] = (int32_t)v;
      return ORC_OK;
    case POKE_STAMP:
      if (i >= p->B) return ORC_EINVAL;
      src->stamps[i] = (uint32_t)v;
      return ORC_OK;
    case POKE_PAGE_SLOT:
      if (i >= p->pages_max) return ORC_EINVAL;
      src->page_slot[i] = (int32_t)v;
      return ORC_OK;
    case POKE_BACKED:
      if (i >= p->pages_max) return ORC_EINVAL;
      src->backed[i] = (uint8_t)v;
      return ORC_OK;
    case POKE_PEND:
      if (i >= p->pages_max) return ORC_EINVAL;
      src->pend[i] = (uint64_t)v;
      return ORC_OK;
    case POKE_SLOT_PAIR:
      if (i >= p->capacity) return ORC_EINVAL;
      p->slot_pair[i] = (int32_t)v;
      return ORC_OK;
    case POKE_SLOT_PAGE:
      if (i >= p->capacity) return ORC_EINVAL;
      p->slot_page[i] = (int32_t)v;
      return ORC_OK;
    case POKE_HOST:
      if (!src->host || i >= p->max_rows * (int64_t)p->E) return ORC_EINVAL;
      src->host[i] = (uint16_t)v;
      return ORC_OK;
    default:
      return ORC_EINVAL;
  }
}
