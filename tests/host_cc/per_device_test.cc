// Host-logic test of the per-device cache used for function attributes,
// occupancy answers and symbol addresses: one value per device id, each
// computed once, ids outside the table never cached.
#include <cstdio>

#include "per_device.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::printf("FAIL line %d: %s\n", __LINE__, #c);        \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  dv::PerDevice cache;
  int calls = 0;
  auto value_for = [&](int dev) { return cache.get(dev, [&] { ++calls; return 100 + dev; }); };

  CHECK(!cache.known(0) && !cache.known(1));
  CHECK(value_for(0) == 100 && calls == 1);
  CHECK(value_for(0) == 100 && calls == 1);   // cached for device 0
  CHECK(!cache.known(1));                     // ... but not for device 1
  CHECK(value_for(1) == 101 && calls == 2);   // device 1 computes its own value
  CHECK(value_for(1) == 101 && calls == 2);
  CHECK(value_for(dv::kMaxDevices - 1) == 100 + dv::kMaxDevices - 1 && calls == 3);
  CHECK(value_for(-1) == 99 && calls == 4);   // unknown device: computed every time
  CHECK(value_for(-1) == 99 && calls == 5);
  CHECK(value_for(dv::kMaxDevices) == 100 + dv::kMaxDevices && calls == 6);
  CHECK(value_for(dv::kMaxDevices) == 100 + dv::kMaxDevices && calls == 7);

  // a computed value equal to a failure code is cached like any other
  dv::PerDevice errs;
  int n = 0;
  CHECK(errs.get(3, [&] { ++n; return 7; }) == 7 && errs.get(3, [&] { ++n; return 0; }) == 7 && n == 1);
  std::printf("ok\n");
  return 0;
}
