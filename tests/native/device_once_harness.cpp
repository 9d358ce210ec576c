// Host test of PerDeviceOnce (the per-device shared-memory opt-in record of
// the tcgen05 launchers): the set-up runs once per device id, again after a
// failure, never for an id outside the table, and exactly once when many
// threads launch on one device at the same time.  Prints one count per line.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "device_once.h"

int main() {
  ulysses::PerDeviceOnce<4> once;
  int calls[4] = {0, 0, 0, 0};
  auto ok = [&](int d) { return [&calls, d]() { ++calls[d]; return 0; }; };
  int rc = 0;
  rc |= once.run(0, ok(0), 99);
  rc |= once.run(0, ok(0), 99);
  rc |= once.run(1, ok(1), 99);
  rc |= once.run(0, ok(0), 99);
  rc |= once.run(1, ok(1), 99);
  // a failing set-up is reported and retried on the next call
  const int fail1 = once.run(2, [&]() { ++calls[2]; return 7; }, 99);
  const int fail2 = once.run(2, [&]() { ++calls[2]; return 7; }, 99);
  const int good = once.run(2, ok(2), 99);
  const int after = once.run(2, ok(2), 99);
  const int range_hi = once.run(4, ok(0), 99);
  const int range_lo = once.run(-1, ok(0), 99);
  // device 3: many threads at once
  std::atomic<int> calls3{0};
  std::vector<std::thread> th;
  for (int t = 0; t < 8; ++t)
    th.emplace_back([&]() {
      for (int i = 0; i < 2000; ++i) once.run(3, [&]() { calls3.fetch_add(1); return 0; }, 99);
    });
  for (auto& x : th) x.join();
  std::printf("rc %d\n", rc);
  std::printf("dev0 %d\ndev1 %d\ndev2 %d\n", calls[0], calls[1], calls[2]);
  std::printf("fail %d %d good %d after %d\n", fail1, fail2, good, after);
  std::printf("range %d %d\n", range_hi, range_lo);
  std::printf("dev3 %d\n", calls3.load());
  return 0;
}
