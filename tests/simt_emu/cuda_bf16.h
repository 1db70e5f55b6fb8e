// Stand-in for the bfloat16 header under the host emulation: storage as the
// upper 16 bits of a float, conversions rounding to nearest even.
#pragma once
#include "emu.h"
struct __nv_bfloat16 {
  uint16_t x;
};
struct __nv_bfloat162 {
  __nv_bfloat16 x, y;
};
inline __nv_bfloat16 __float2bfloat16_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) != 0x7f800000u) u = u + 0x7fffu + ((u >> 16) & 1u);
  else if (u & 0x007fffffu) u |= 0x00400000u;
  __nv_bfloat16 b;
  b.x = (uint16_t)(u >> 16);
  return b;
}
inline float __bfloat162float(__nv_bfloat16 b) {
  uint32_t u = (uint32_t)b.x << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
inline __nv_bfloat16 __ushort_as_bfloat16(unsigned short s) { __nv_bfloat16 b; b.x = s; return b; }
inline unsigned short __bfloat16_as_ushort(__nv_bfloat16 b) { return b.x; }

inline float2 __bfloat1622float2(__nv_bfloat162 v) { return make_float2(__bfloat162float(v.x), __bfloat162float(v.y)); }
inline __nv_bfloat162 __floats2bfloat162_rn(float a, float b) { return __nv_bfloat162{__float2bfloat16_rn(a), __float2bfloat16_rn(b)}; }
