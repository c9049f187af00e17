// Compile-time dispatch on the padded state count NT in {4, 8, 16, 32, 64}.
#pragma once

#define SSK_DISPATCH_NT(N, ...)              \
  do {                                        \
    if ((N) <= 4) { constexpr int NT = 4; __VA_ARGS__; }        \
    else if ((N) <= 8) { constexpr int NT = 8; __VA_ARGS__; }   \
    else if ((N) <= 16) { constexpr int NT = 16; __VA_ARGS__; } \
    else if ((N) <= 32) { constexpr int NT = 32; __VA_ARGS__; } \
    else if ((N) <= 64) { constexpr int NT = 64; __VA_ARGS__; } \
    else return -1;                           \
  } while (0)
