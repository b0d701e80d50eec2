// The chunk preparation kernel with claimed work items (PrepRange::counter):
// each CTA takes chunks from a counter instead of a fixed persistent stride,
// for the pipelined forward. Same source as chunk_prep.cu, compiled as its own
// translation unit.
#define GDR_PREP_CLAIMED
#include "chunk_prep.cu"
