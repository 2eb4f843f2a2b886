// Launch shape of the decode pass, shared by the host code that sizes the split count
// and workspace and by the launcher, so that both always agree.
#pragma once

namespace fa {

// Two shapes of fa_decode_kernel at d = 128:
//  * default: two CTAs per SM, each with a K/V ring of 2 tiles (one 128-key block), and
//    as many key splits as fill 304 CTA slots;
//  * deep ring: one CTA per SM with a ring of 4 tiles (two blocks in flight), and as
//    many splits as fill 152 SMs.
// Measured on GB300 (Hq = 32, Hkv = 8, d = 128, one new query): the deep ring is 3-5%
// faster when there are at most 8 (batch, kv head) units, where the default needs twice
// as many splits (B = 1 x 65536 keys: 5017 against 4764 GB/s; B = 1 x 131072: 5933
// against 5744), level at 16 units, and slower above (32 units: 4544 against 4697;
// 256 units no longer fit one wave).
inline bool decode_deep_ring(int d, long long units) { return d == 128 && units <= 8; }

inline int decode_cta_slots(int d, long long units) { return decode_deep_ring(d, units) ? 152 : 304; }

}  // namespace fa
