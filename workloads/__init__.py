"""Seeded synthetic inputs of the MoE layer workloads (shared by the tests, bench.py and smoke()).

Random draws and shapes only: none of the method's arithmetic lives here.
"""
