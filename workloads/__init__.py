"""Seeded synthetic input generators shared by the tests, the bench and the oracle checks."""
