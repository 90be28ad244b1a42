// Host-side probe of the library's host logic, run without a GPU by
// tests/test_host_logic.py. Reads commands from stdin, one result per line:
//   k <tau> <n>                                  -> keep_count(tau, n)
//   s <units> <len> <max_splits> <num_sms> <active[1..16]>
//                                                -> choose_splits(...)
#include <stdio.h>

#include "attend_kernels.cuh"

int main() {
  char cmd[4];
  while (scanf("%3s", cmd) == 1) {
    if (cmd[0] == 'k') {
      double tau;
      int n;
      if (scanf("%lf %d", &tau, &n) != 2) return 2;
      printf("%d\n", fastocr::keep_count(tau, n));
    } else if (cmd[0] == 's') {
      long units, len;
      int max_splits, num_sms, active[fastocr::kMaxSplits + 1] = {0};
      if (scanf("%ld %ld %d %d", &units, &len, &max_splits, &num_sms) != 4) return 2;
      for (int s = 1; s <= fastocr::kMaxSplits; ++s)
        if (scanf("%d", &active[s]) != 1) return 2;
      printf("%d\n", fastocr::choose_splits(units, len, max_splits, active, num_sms));
    } else {
      return 2;
    }
  }
  return 0;
}
