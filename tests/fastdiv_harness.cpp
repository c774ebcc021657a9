// Prints the multiply-shift constants the library derives for each divisor
// given on the command line: "d m s one" per line (host code of launch.h).
#include <cstdio>
#include <cstdlib>

#include "launch.h"

int main(int argc, char **argv)
{
    for (int i = 1; i < argc; ++i) {
        const unsigned long d = std::strtoul(argv[i], nullptr, 10);
        const vq::FastDiv f = vq::make_fastdiv((uint32_t)d);
        std::printf("%lu %u %u %u\n", d, f.m, f.s, f.one);
    }
    return 0;
}
