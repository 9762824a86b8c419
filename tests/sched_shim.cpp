// Test shim: exposes the kernels' work schedule (schedule.h, compiled here as
// plain C++) so the CPU tests can enumerate every unit each slot would run.
#include "schedule.h"

extern "C" {

static g10::Sched make(const int64_t* p) {
  g10::Sched s;
  s.tiles_i = static_cast<int32_t>(p[0]);
  s.tiles_j = static_cast<int32_t>(p[1]);
  s.num_kb = static_cast<int32_t>(p[2]);
  s.raster_group = static_cast<int32_t>(p[3]);
  s.mode = static_cast<int32_t>(p[4]);
  s.split_k = static_cast<int32_t>(p[5]);
  s.dp_tiles = static_cast<int32_t>(p[6]);
  s.sk_slots = static_cast<int32_t>(p[7]);
  s.sk_iters = p[8];
  s.batch = static_cast<int32_t>(p[9]);
  s.groups = 0;
  s.group_tile_start = nullptr;
  return s;
}

static const int32_t* g_table = nullptr;  // grouped schedules: tile prefix of the current call
static int32_t g_groups = 0;

static g10::Sched make_any(const int64_t* p) {
  g10::Sched s = make(p);
  s.groups = g_groups;
  s.group_tile_start = g_table;
  return s;
}

// Set (or clear, groups = 0) the group table used by the calls below.
void sched_set_groups(const int32_t* table, int32_t groups) {
  g_table = table;
  g_groups = groups;
}

// Units of `slot` (of `slots`), 12 int32 each:
// ti tj tile kb0 kb1 partial pslot ctr ncontrib first_c first_j tb.
int sched_units(const int64_t* params, int32_t slot, int32_t slots, int32_t* out, int32_t cap) {
  const g10::Sched s = make_any(params);
  g10::WorkIter it(s, slot, slots);
  g10::Unit w;
  int n = 0;
  while (it.next(w)) {
    if (n < cap) {
      int32_t* o = out + 12 * n;
      o[0] = w.ti; o[1] = w.tj; o[2] = w.tile; o[3] = w.kb0; o[4] = w.kb1; o[5] = w.partial;
      o[6] = w.pslot; o[7] = w.ctr; o[8] = w.ncontrib; o[9] = w.first_c; o[10] = w.first_j;
      o[11] = w.tb;
    }
    ++n;
  }
  return n;
}

// contrib_slot() for a unit given as the 12 fields above.
int32_t sched_contrib_slot(const int64_t* params, const int32_t* u, int32_t k) {
  const g10::Sched s = make_any(params);
  g10::Unit w;
  w.ti = u[0]; w.tj = u[1]; w.tile = u[2]; w.kb0 = u[3]; w.kb1 = u[4]; w.partial = u[5];
  w.pslot = u[6]; w.ctr = u[7]; w.ncontrib = u[8]; w.first_c = u[9]; w.first_j = u[10];
  w.tb = u[11];
  return g10::contrib_slot(s, w, k);
}

int64_t sched_partial_slots(const int64_t* params) { return g10::partial_slots(make_any(params)); }

}
