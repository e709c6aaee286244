/*
 * mla_debug.h -- test hooks of the MLA decode library.  They are not part of
 * the decode API in mla.h and exist so that tests can drive code paths the
 * problem size alone does not choose.
 */
#ifndef MLA_DEBUG_H_
#define MLA_DEBUG_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Limit the number of two-SM CTA pairs (with at most 16 heads, where one
 * CTA per SM takes a pair's place: the number of CTAs) over which the
 * tensor-core path of mla_decode (and mla_decode_noalloc) cuts its split
 * plan: every later call in this process lays the items' tiles end to end
 * and cuts them into at most `pairs` equal ranges, so an item is cut into
 * more or fewer pieces than the full GPU would cut it.  pairs <= 0 removes
 * the limit (every co-resident pair, or every SM, takes part, the
 * default).  Returns the previous limit
 * (0 = none).  The result of mla_decode does not depend on the split beyond
 * fp32 rounding, which is what the split-invariance tests check; the limit
 * is process-wide, so set it only where no other thread decodes. */
int mla_debug_set_decode_pairs(int pairs);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DEBUG_H_ */
