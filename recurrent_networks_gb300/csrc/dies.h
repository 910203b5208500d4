// The grid kernels' die placement: its decisions from measured L2 round
// trips, host only (csrc/dies.cu), shared by the placement itself and by the
// what-if entry point rnn_die_plan_for.
#pragma once

namespace rnn {

// The split point of two latency clusters (0: a fast/slow ratio under 1.3,
// not trusted); each SM's die (entry 0 is the measuring CTA, on die 0) with
// the count per die; each 1 KB block's home die (-1 for all when the split is
// not trusted); the number of batch groups of C CTAs on die 0 (the split
// closest to even that fits, or -1); and each group's counter word in the
// first free block homed on its die (groups below g0 on die 0).
unsigned long long split_point(const unsigned long long* v, int n);
bool classify_sms(const unsigned long long* lat, int n, signed char* die, int count[2]);
bool classify_blocks(const unsigned long long* lat, int n, signed char* home);
int die_split_groups(int groups, int C, const int cnt[2]);
bool die_assign_counters(int groups, int g0, const signed char* home, int nblocks, int* ctr_word);

}  // namespace rnn
