"""Planted mistakes in the oracle must each fail at least one pin (no GPU).

Each case copies ``oracle/grid_oracle.c``, changes one statement the way a
plausible slip would (a wrong sign, a dropped term, a transposed stride, an
off-by-one clamp, the wrong gather direction ...), compiles the copy and runs
every pin against it in a child process.  The pins are trustworthy only if
none of these mutants gets through.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "origin_sign": ("float t = p - o;", "float t = p + o;"),
    "dropped_invcell": ("float u = t * invCell;", "float u = t;"),
    "floor_to_round": ("float f = floorf(u);", "float f = roundf(u);"),
    "clamp_off_by_one": ("return dim - 1u;", "return dim - 2u;"),
    "transposed_stride": ("return x + y * gx + z * gx * gy;", "return x + y * gy + z * gx * gy;"),
    "z_stride_dropped": ("return x + y * gx + z * gx * gy;", "return x + y * gx + z * gy;"),
    "wrong_origin_axis": ("axis_cell(pos[1], origin[1]", "axis_cell(pos[1], origin[0]"),
    "wrong_position_axis": ("axis_cell(pos[2], origin[2]", "axis_cell(pos[1], origin[2]"),
    "histogram_set_not_add": ("conteos[celdaDe[i]] += 1u;", "conteos[celdaDe[i]] = 1u;"),
    "scan_dropped_term": ("inicios[c + 1] = inicios[c] + conteos[c];", "inicios[c + 1] = conteos[c];"),
    "scan_inclusive": ("inicios[0] = 0u;", "inicios[0] = cells ? conteos[0] : 0u;"),
    "cursor_not_advanced": ("cursor[c] = slot + 1u;", "cursor[c] = slot;"),
    "reversed_within_cell": ("ordenado[inicios[c] + slot] = (uint32_t)i;",
                             "ordenado[inicios[c + 1] - 1u - slot] = (uint32_t)i;"),
    "scatter_direction_reorder": (
        "memcpy(dst + ORACLE_RECORD_BYTES * k, src + ORACLE_RECORD_BYTES * (uint64_t)ordenado[k],",
        "memcpy(dst + ORACLE_RECORD_BYTES * (uint64_t)ordenado[k], src + ORACLE_RECORD_BYTES * k,"),
    "overflow_off_by_one": ("if (previo + 1u > capacidad)", "if (previo > capacidad)"),
    "max_of_previo": ("            diag[0] = previo + 1u;", "            diag[0] = previo;"),
    "records_scatter_direction": ("memcpy(dst + (uint64_t)record_bytes * k, src + (uint64_t)record_bytes * ordenado[k], record_bytes);",
                                  "memcpy(dst + (uint64_t)record_bytes * ordenado[k], src + (uint64_t)record_bytes * k, record_bytes);"),
    "stencil_one_sided": ("for (int dz = -1; dz <= 1; ++dz) {", "for (int dz = -1; dz <= 0; ++dz) {"),
    "radius_not_squared": ("if (r2 < h2) {", "if (r2 < h) {"),
    "own_mass": ("sum += (double)pj[7] * t * t * t;", "sum += (double)pi[7] * t * t * t;"),
    "half_record_copied": ("               ORACLE_RECORD_BYTES);", "               ORACLE_RECORD_BYTES / 2);"),
    "morton_x_bit_from_y": ("if (l < bits[0]) code |= ((x >> l) & 1u) << pos++;",
                            "if (l < bits[0]) code |= ((y >> l) & 1u) << pos++;"),
    "morton_position_not_advanced": ("if (l < bits[2]) code |= ((z >> l) & 1u) << pos++;",
                                     "if (l < bits[2]) code |= ((z >> l) & 1u) << pos;"),
    "morton_y_before_x": ("if (l < bits[1]) code |= ((y >> l) & 1u) << pos++;",
                          "if (l < bits[1]) code |= ((y >> l) & 1u) << (pos++ - 1u);"),
    "morton_bits_rounded_up": ("while ((1u << b) < d)", "while ((1u << b) <= d)"),
    "morton_shared_bit_count": ("log2_exact(dims[1]), log2_exact(dims[2])", "log2_exact(dims[0]), log2_exact(dims[2])"),
    "order_ignored_by_count": ("celdaDe[i] = cell_in_order(x, y, z, dims, order);",
                               "celdaDe[i] = cell_in_order(x, y, z, dims, 0u);"),
    "order_ignored_by_density": ("(uint32_t)z, dims, order);", "(uint32_t)z, dims, 0u);"),
    "upper_clamp_strict": ("if ((double)f >= (double)dim)", "if ((double)f > (double)dim)"),
    "below_clamped_to_top": ("    if (isnan(f) || f < 0.0f)\n        return 0u;", "    if (isnan(f) || f < 0.0f)\n        return dim - 1u;"),
    "density_square_not_cube": ("sum += (double)pj[7] * t * t * t;", "sum += (double)pj[7] * t * t;"),
    "density_x_one_sided": ("for (int dx = -1; dx <= 1; ++dx) {", "for (int dx = 0; dx <= 1; ++dx) {"),
    "density_y_against_x": ("const double ey = (double)pj[1] - (double)pi[1];",
                            "const double ey = (double)pj[1] - (double)pi[0];"),
    "canonical_pairs_left_unsorted": ("if (b > a + 1u)", "if (b > a + 2u)"),
    "records_fixed_stride": ("src + (uint64_t)record_bytes * ordenado[k], record_bytes);",
                             "src + (uint64_t)32u * ordenado[k], record_bytes);"),
}

RUNNER = """
import sys
sys.path[:0] = [{root!r}, {here!r}]
import oracle, pins
o = oracle.Oracle({lib!r})
for pin in pins.ALL_PINS:
    try:
        pin(o)
    except AssertionError as e:
        print("CAUGHT", pin.__name__, str(e)[:200])
        sys.exit(3)
print("ESCAPED")
sys.exit(0)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as fh:
        src = fh.read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = str(tmp_path / "libmutant.so")
    oracle.compile_oracle(str(mutated), lib)
    proc = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, here=HERE, lib=lib)],
                          capture_output=True, text=True, timeout=300)
    assert "ESCAPED" not in proc.stdout, f"mutant {name} passed every pin"
    assert proc.returncode == 3 and "CAUGHT" in proc.stdout, (
        f"mutant {name} did not fail a pin cleanly: rc={proc.returncode}\n{proc.stdout}\n{proc.stderr[-2000:]}")
