/* Calls the library through its C header from plain C99: no CUDA headers, no C++, no device
 * needed for these calls (version, status strings, argument validation before any launch). */
#include <stdio.h>
#include <string.h>

#include "fa.h"

int main(void) {
  const int v = fa_abi_version();
  printf("abi %d.%d\n", v >> 16, v & 0xffff);
  if (v >> 16 != 2) return 1;
  printf("status0 %s\n", fa_status_string(0));
  /* a null q pointer is an invalid argument, reported before anything is launched */
  const int st = fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 64, 0.125f, 0, NULL);
  printf("null-args %d %s\n", st, fa_status_string(st));
  if (st != 1) return 2;
  /* fp32 forward: an unsupported head dimension (rejected before the pointers are looked at
   * beyond being non-null) */
  float dummy[4];
  const int st2 = fa_fwd_fp32(dummy, dummy, dummy, dummy, dummy, 1, 1, 4, 48, 0.125f, 0, NULL);
  if (st2 != 2) return 3;
  return 0;
}
