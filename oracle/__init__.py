"""Float64 CPU oracle of the sparse-MoE forward layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check of the
package entry file and by the CPU-baseline / reference legs of the benchmark
script; never by the library.
"""
