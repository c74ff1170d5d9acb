"""The CTA-order mapping (csrc/grid_order.cuh) on the host: every CTA index
of a grid over (plane, block) pairs maps to a distinct pair, all pairs are
covered, and inside each group of planes the ranks never decrease with the
index (each group's longest blocks start first)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r'''
#include <cstdio>
#include <vector>
#include "grid_order.cuh"
int main() {
    const int sms_list[] = {1, 7, 152};
    int bad = 0, cases = 0;
    for (int planes = 1; planes <= 40; planes += 3)
        for (int blocks = 1; blocks <= 70; blocks += 7)
            for (int sms : sms_list) {
                const int group = fa::grid_group_planes(planes, blocks, sms);
                if (group < 1 || group > planes) ++bad;
                std::vector<int> seen(planes * blocks, 0);
                int prev_grp = -1, prev_rank = -1;
                for (int idx = 0; idx < planes * blocks; ++idx) {
                    int plane = -1, rank = -1;
                    fa::grid_decode(idx, planes, blocks, group, plane, rank);
                    if (plane < 0 || plane >= planes || rank < 0 || rank >= blocks) { ++bad; continue; }
                    seen[plane * blocks + rank]++;
                    const int grp = plane / group;
                    if (grp == prev_grp && rank < prev_rank) ++bad;
                    if (grp < prev_grp) ++bad;
                    prev_grp = grp;
                    prev_rank = rank;
                }
                for (int v : seen) if (v != 1) ++bad;
                ++cases;
            }
    printf("%d %d\n", cases, bad);
    return 0;
}
'''


def test_grid_decode_is_a_grouped_bijection(tmp_path):
    from exact_attention_85_gb300 import build
    src = tmp_path / "grid_order_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "grid_order_check"
    inc = os.path.join(ROOT, "exact_attention_85_gb300", "csrc")
    r = subprocess.run([build._nvcc(), "-std=c++17", "-I", inc, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    cases, bad = map(int, out.stdout.split())
    assert cases > 0 and bad == 0
