// walk.cuh -- iterate the segments of one CTA's page range.
//
// Pages are ordered (b, kvh, page).  A CTA owns [cta_start[c], cta_start[c+1])
// of that order; a segment is the part of one unit (b, kvh) inside it.  The
// producer and consumer warps walk the same segments in the same order.
#pragma once

#include "common.cuh"

namespace kv {

struct Seg {
  int b, kvh, j0, j1;  // unit and page range [j0, j1)
  int n;               // pages of the whole unit
  bool full;           // the segment is the whole unit
};

KV_DEVI bool pos_less(int4 a, int4 b) {
  return a.x < b.x || (a.x == b.x && (a.y < b.y || (a.y == b.y && a.z < b.z)));
}

struct Walker {
  const int64_t* cum;
  int units_per_seq;
  int4 cur, end;

  KV_DEVI bool next(Seg& s) {
    while (pos_less(cur, end)) {
      const int n = int(cum[cur.x + 1] - cum[cur.x]);
      if (n == 0 || cur.z >= n) {
        advance();
        continue;
      }
      const int j1 = (cur.x == end.x && cur.y == end.y) ? end.z : n;
      s.b = cur.x;
      s.kvh = cur.y;
      s.j0 = cur.z;
      s.j1 = j1;
      s.n = n;
      s.full = (cur.z == 0 && j1 == n);
      advance();
      return true;
    }
    return false;
  }

  KV_DEVI void advance() {
    cur.z = 0;
    if (++cur.y == units_per_seq) {
      cur.y = 0;
      ++cur.x;
    }
  }
};

}  // namespace kv
