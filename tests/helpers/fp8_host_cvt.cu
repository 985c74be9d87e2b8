// Host-side reference for the FP8 E4M3 encoder pin: reads float32 values from
// the file argv[1], converts each with CUDA's own host implementation of
// __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3) (round to nearest even,
// saturating to +-448) and writes one code byte per value to argv[2].
// It runs on the CPU only; no device code is involved.
#include <cuda_fp8.h>

#include <cstdio>
#include <vector>

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* in = std::fopen(argv[1], "rb");
  if (!in) return 3;
  std::vector<float> xs;
  float x;
  while (std::fread(&x, sizeof(float), 1, in) == 1) xs.push_back(x);
  std::fclose(in);
  std::vector<unsigned char> out(xs.size());
  for (size_t i = 0; i < xs.size(); ++i)
    out[i] = static_cast<unsigned char>(__nv_cvt_float_to_fp8(xs[i], __NV_SATFINITE, __NV_E4M3));
  FILE* o = std::fopen(argv[2], "wb");
  if (!o) return 4;
  std::fwrite(out.data(), 1, out.size(), o);
  std::fclose(o);
  return 0;
}
