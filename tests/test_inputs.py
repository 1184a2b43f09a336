"""The seeded generators' storage conversions (shared by the oracle side and the
GPU side of the tests) against the formats' definitions."""
import numpy as np

from video_dit_long_gb300 import inputs


def test_e4m3_codes_round_trip():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]  # the two NaN codes
    v = inputs.e4m3_to_f32(codes)
    back = inputs.e4m3_bits(v)
    # every finite code widens and rounds back to itself (+0 and -0 are both zero)
    same = (back == codes) | ((codes & 0x7F) == 0) & ((back & 0x7F) == 0)
    assert same.all()


def test_e4m3_known_values_and_rounding():
    # largest finite 1.75 * 2^8, smallest normal 2^-6, smallest subnormal 2^-9
    assert inputs.e4m3_to_f32(np.array([0x7E, 0x08, 0x01, 0x38, 0xB8], np.uint8)).tolist() == \
        [448.0, 2.0**-6, 2.0**-9, 1.0, -1.0]
    # 1 + 1/16 lies halfway between 1 (code 0x38, even) and 1.125 (0x39): ties go to the even code
    assert inputs.e4m3_bits(np.array([1.0625, 1.1875], np.float32)).tolist() == [0x38, 0x3A]
    # beyond the range: saturates at +-448
    assert inputs.e4m3_bits(np.array([1e4, -600.0], np.float32)).tolist() == [0x7E, 0xFE]
    # nearest: 0.3 lies between 0.28125 and 0.3125
    assert inputs.e4m3_to_f32(inputs.e4m3_bits(np.array([0.3], np.float32)))[0] == 0.3125


def test_e4m3_error_bound():
    x = inputs.normal_f32(3, 1, 100000)
    y = inputs.e4m3_to_f32(inputs.e4m3_bits(x)).astype(np.float64)
    err = np.abs(y - x)
    # half a unit in the last place: 2^-4 relative for normals, 2^-10 absolute below 2^-6
    assert (err <= np.maximum(np.abs(x) * 2.0**-4, 2.0**-10) * (1 + 1e-12)).all()
